"""The C ABI without a GPU: the library loads, exports every entry point that
include/wq.h declares, and rejects invalid arguments on the host before it
touches a device.  Only arguments that fail validation are passed, with
placeholder pointers that are never dereferenced."""
import ctypes
import os
import re

import pytest

from weight_only_quantized_wq_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000  # 16-byte aligned placeholder, never dereferenced (validation fails first)


@pytest.fixture(scope="module")
def L():
    from weight_only_quantized_wq_gb300 import build
    build.build()
    return binding.lib()


def declared():
    src = open(os.path.join(ROOT, "include", "wq.h")).read()
    return re.findall(r"WQ_API[^;(]*?\b(wq_\w+)\s*\(", src)


def test_header_declares_expected_entry_points():
    assert set(declared()) == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared():
        assert hasattr(L, name), name
        assert isinstance(getattr(L, name), ctypes._CFuncPtr)
    src = open(os.path.join(ROOT, "include", "wq_testing.h")).read()
    testing = re.findall(r"WQ_API[^;(]*?\b(wq_\w+)\s*\(", src)
    assert set(testing) == set(binding.TESTING_EXPORTS)
    for name in testing:
        assert hasattr(L, name), name


def test_testing_hook_validates_on_the_host(L):
    S = {n: i for i, n in enumerate(binding.STATUS)}
    f = L.wq_testing_decode_timeout
    args = [FAKE, 1, FAKE, FAKE, 1, None, 4, 64, 128, 4, 64, FAKE, None, 0]
    assert f(*args, 100, 1, None) == S["WQ_ERR_SHAPE"]            # limit too short
    assert f(*args, 10 ** 10, 1, None) == S["WQ_ERR_SHAPE"]       # limit too long
    assert f(*args, 100000, -1, None) == S["WQ_ERR_SHAPE"]        # no stage withheld
    args[6] = 65
    assert f(*args, 100000, 1, None) == S["WQ_ERR_SHAPE"]         # not the few-token kernel
    args[6] = 4
    args[0] = FAKE + 2
    assert f(*args, 100000, 1, None) == S["WQ_ERR_ALIGN"]


def test_status_strings(L):
    for i in range(len(binding.STATUS)):
        assert binding.wq_status_string(i)
    assert binding.wq_status_string(99) == "unknown status"


def test_sizes(L):
    assert binding.wq_chunk_k(4) == 64 and binding.wq_chunk_k(2) == 128 and binding.wq_chunk_k(8) == 32
    assert binding.wq_chunk_k(3) == 0
    assert binding.wq_packed_bytes(4096, 11008, 4) == 4096 * 11008 // 2
    assert binding.wq_packed_bytes(8192, 8192, 2) == 8192 * 8192 // 4
    assert binding.wq_packed_bytes(4096, 4096, 8) == 4096 * 4096
    assert binding.wq_packed_bytes(100, 64, 4) == 0   # K not a multiple of 64
    assert binding.wq_packed_bytes(64, 20, 4) == 0    # N not a multiple of 16
    assert binding.wq_packed_bytes(64, 16, 3) == 0


def _mm(L, **kw):
    a = dict(x=FAKE, xd=1, w=FAKE, s=FAKE, sd=1, z=None, M=4, N=64, K=128, wb=4, gs=64, out=FAKE, ws=None, wsb=0)
    a.update(kw)
    return L.wq_matmul(a["x"], a["xd"], a["w"], a["s"], a["sd"], a["z"], a["M"], a["N"], a["K"], a["wb"], a["gs"],
                       a["out"], a["ws"], a["wsb"], None)


def test_matmul_ex_host_validation(L):
    S = {n: i for i, n in enumerate(binding.STATUS)}

    def mx(odt, **kw):
        a = dict(x=FAKE, xd=1, w=FAKE, s=FAKE, sd=1, z=None, M=4, N=64, K=128, wb=4, gs=64, out=FAKE + 8)
        a.update(kw)
        return L.wq_matmul_ex(a["x"], a["xd"], a["w"], a["s"], a["sd"], a["z"], a["M"], a["N"], a["K"], a["wb"],
                              a["gs"], a["out"], odt, None, 0, None)
    assert mx(3) == S["WQ_ERR_DTYPE"]      # no such output type
    assert mx(-1) == S["WQ_ERR_DTYPE"]
    assert mx(0) == S["WQ_ERR_ALIGN"]      # a valid type reaches the alignment check (out misaligned)
    assert mx(1, out=None) == S["WQ_ERR_NULL"]
    assert mx(1, M=0) == S["WQ_OK"]


def test_matmul_host_validation(L):
    S = {n: i for i, n in enumerate(binding.STATUS)}
    assert _mm(L, x=None) == S["WQ_ERR_NULL"]
    assert _mm(L, out=None) == S["WQ_ERR_NULL"]
    assert _mm(L, wb=3) == S["WQ_ERR_WBIT"]
    assert _mm(L, K=0) == S["WQ_ERR_SHAPE"]
    assert _mm(L, M=-1) == S["WQ_ERR_SHAPE"]
    assert _mm(L, N=40) == S["WQ_ERR_SHAPE"]
    assert _mm(L, K=96) == S["WQ_ERR_SHAPE"]
    assert _mm(L, xd=2) == S["WQ_ERR_DTYPE"]
    assert _mm(L, sd=2) == S["WQ_ERR_DTYPE"]
    assert _mm(L, wb=8, sd=1) == S["WQ_ERR_DTYPE"]
    assert _mm(L, wb=8, sd=2, z=FAKE) == S["WQ_ERR_DTYPE"]
    assert _mm(L, gs=48) == S["WQ_ERR_GROUP"]
    assert _mm(L, gs=8) == S["WQ_ERR_GROUP"]
    assert _mm(L, gs=0) == S["WQ_ERR_GROUP"]
    assert _mm(L, x=FAKE + 8) == S["WQ_ERR_ALIGN"]
    assert _mm(L, out=FAKE + 4) == S["WQ_ERR_ALIGN"]
    assert _mm(L, w=FAKE + 2) == S["WQ_ERR_ALIGN"]
    # M == 0 and N == 0 are no-ops that succeed without touching a device
    assert _mm(L, M=0) == S["WQ_OK"]
    assert _mm(L, N=0) == S["WQ_OK"]


def test_pack_host_validation(L):
    S = {n: i for i, n in enumerate(binding.STATUS)}
    assert L.wq_pack(None, 64, 16, 4, FAKE, None) == S["WQ_ERR_NULL"]
    assert L.wq_pack(FAKE, 64, 16, 5, FAKE, None) == S["WQ_ERR_WBIT"]
    assert L.wq_pack(FAKE, 60, 16, 4, FAKE, None) == S["WQ_ERR_SHAPE"]
    assert L.wq_pack(FAKE, 64, 8, 4, FAKE, None) == S["WQ_ERR_SHAPE"]
    assert L.wq_pack(FAKE + 4, 64, 16, 4, FAKE, None) == S["WQ_ERR_ALIGN"]
    assert L.wq_unpack(FAKE, 64, 16, 4, None, None) == S["WQ_ERR_NULL"]
    assert L.wq_unpack(FAKE, 0, 16, 4, FAKE, None) == S["WQ_ERR_SHAPE"]


def test_workspace_bytes_invalid_is_zero(L):
    assert binding.wq_workspace_bytes(0, 64, 128, 4, 64) == 0
    assert binding.wq_workspace_bytes(4, 64, 100, 4, 64) == 0


def test_binding_marshals_to_the_c_abi_and_raises_its_status():
    # CPU tensors and a stand-in stream: the call crosses ctypes and the C side
    # rejects it with a status, which the binding raises as WQError.  x is a
    # view two bytes into its buffer, so the alignment check of wq_matmul
    # (which runs before any device query or launch) returns WQ_ERR_ALIGN on
    # every machine, with or without a GPU: nothing is ever launched on these
    # host pointers.
    import torch
    from weight_only_quantized_wq_gb300 import binding

    class Stream:
        cuda_stream = 0

    xbuf = torch.zeros(1, 512 + 8, dtype=torch.bfloat16)
    x = xbuf[:, 1:513]
    assert x.data_ptr() % 16 == 2
    q = torch.zeros(512 * 512 // 2, dtype=torch.uint8)
    s = torch.zeros(4, 512, dtype=torch.bfloat16)
    out = torch.zeros(1, 512)
    with pytest.raises(binding.WQError) as e:
        binding.wq_matmul(x, q, s, None, 1, 512, 512, 4, 128, out=out, stream=Stream())
    assert e.value.status == binding.STATUS.index("WQ_ERR_ALIGN")
    with pytest.raises(binding.WQError) as e:
        binding.wq_matmul_noalloc(x, q, s, None, 1, 512, 512, 4, 128, out=out, stream=Stream())
    assert e.value.status == binding.STATUS.index("WQ_ERR_ALIGN")


def test_matmul_path_rules(L):
    # the path is a host decision (no device): few tokens or codes / groups the
    # tensor-core kernels do not take -> 0; int4 with 64-aligned groups -> 1
    # (exact); many tokens where rounding w once holds the bound -> 2; bf16
    # below K = 4096 on grids of at least 128 tiles -> 3 (two-term weights)
    F16, BF16, F32 = binding.WQ_F16, binding.WQ_BF16, binding.WQ_F32
    P = binding.wq_matmul_path
    N = 4096
    assert P(16, N, 8192, 4, 128, BF16, BF16) == 0
    assert P(64, N, 8192, 4, 128, BF16, BF16) == 0
    assert P(65, N, 8192, 4, 128, BF16, BF16) == 2
    assert P(4096, N, 8192, 4, 128, BF16, BF16) == 2
    assert P(65, N, 2048, 4, 128, BF16, BF16) == 1     # bf16 below K = 4096: exact path
    assert P(4096, N, 512, 4, 128, F16, F16) == 2      # fp16 rounding holds the bound
    assert P(4096, N, 8192, 4, 128, F16, BF16) == 1    # scale dtype differs from x
    assert P(4096, N, 8192, 4, 32, BF16, BF16) == 0    # group not a multiple of 64
    assert P(4096, N, 8192, 2, 64, BF16, BF16) == 0    # int2
    assert P(64, N, 4096, 8, -1, BF16, F32) == 0       # int8
    assert P(100, N, 4096, 4, -1, BF16, BF16) == 2     # per channel
    assert P(100, N, 2048, 4, -1, BF16, BF16) == 1
    # two-term weights: ceil(M / 256) * ceil(N / 128) >= 128 tiles and M >= 129
    assert P(1024, 4096, 2048, 4, 128, BF16, BF16) == 3   # 4 x 32 tiles
    assert P(768, 4096, 2048, 4, 128, BF16, BF16) == 1    # 3 x 32 tiles
    assert P(256, 16384, 1024, 4, 128, BF16, BF16) == 3   # 1 x 128 tiles
    assert P(128, 28672, 2048, 4, 128, BF16, BF16) == 1   # under 129 tokens
    assert P(1024, 4096, 2048, 4, 128, F16, F16) == 2     # fp16: one rounding holds
    assert P(64, N, 4096, 3, 128, BF16, BF16) == -1
    assert P(64, N, 4096, 4, 48, BF16, BF16) == -1
    assert P(64, N, 4096, 8, -1, BF16, BF16) == -1
    assert P(64, 24, 4096, 4, 128, BF16, BF16) == -1     # N not a multiple of 16
    assert P(64, 0, 4096, 4, 128, BF16, BF16) == -1


def test_t2_host_validation(L):
    S = {n: i for i, n in enumerate(binding.STATUS)}
    assert L.wq_t2_pack(None, 128, 16, FAKE, None) == S["WQ_ERR_NULL"]
    assert L.wq_t2_pack(FAKE, 64, 16, FAKE, None) == S["WQ_ERR_SHAPE"]      # K not a multiple of 128
    assert L.wq_t2_pack(FAKE, 128, 24, FAKE, None) == S["WQ_ERR_SHAPE"]     # N not a multiple of 16
    assert L.wq_t2_pack(FAKE, 65536 + 128, 16, FAKE, None) == S["WQ_ERR_SHAPE"]  # sums could pass 2^24
    assert L.wq_t2_pack(FAKE + 4, 128, 16, FAKE, None) == S["WQ_ERR_ALIGN"]
    mm = L.wq_t2_matmul
    assert mm(None, FAKE, 4, 16, 128, FAKE, FAKE, 1 << 20, None) == S["WQ_ERR_NULL"]
    assert mm(FAKE, FAKE, 4, 16, 100, FAKE, FAKE, 1 << 20, None) == S["WQ_ERR_SHAPE"]
    assert mm(FAKE, FAKE, -1, 16, 128, FAKE, FAKE, 1 << 20, None) == S["WQ_ERR_SHAPE"]
    assert mm(FAKE + 8, FAKE, 4, 16, 128, FAKE, FAKE, 1 << 20, None) == S["WQ_ERR_ALIGN"]
    assert mm(FAKE, FAKE, 0, 16, 128, FAKE, FAKE, 0, None) == S["WQ_OK"]
    assert binding.wq_t2_workspace_bytes(4, 16, 100) == 0
