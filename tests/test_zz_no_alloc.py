"""wq_matmul_noalloc: the entry point for callers that cannot allocate device
memory (it uses a fixed scratch array inside the library instead of a caller
workspace).  Its output must match wq_matmul's, within the tolerance the
other parity tests use, on two calls in a row (the second call reuses the
scratch the first one left behind), and the fp64 oracle's as well.  This file
is collected last on purpose."""
import numpy as np
import pytest
import torch

import weight_only_quantized_wq_gb300 as wq
from weight_only_quantized_wq_gb300 import synthetic as syn
from tests.helpers import assert_close, oracle_y, to_device

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 8 << 20  # the scratch array's size, as include/wq.h states it


def _narrow():
    # One column block over a long K: more K splits than one thread-block
    # cluster reduces, so the partial sums go through the scratch memory.
    return syn.grouped("int4-asym narrow", 4, 8192, 64, 4, 128, "bf16", "bf16", (0.002, 0.02), seed=5)


@pytest.mark.parametrize("make", [_narrow, syn.int4_sym_decode, syn.int2_asym, syn.int8_per_channel],
                         ids=["narrow_long_k", "int4_sym_decode", "int2_asym", "int8_per_channel"])
def test_noalloc_matches_workspace_entry_point_twice(make):
    p = make()
    d = to_device(p)
    need = wq.wq_workspace_bytes(p.M, p.N, p.K, p.w_bit, p.group_size)
    ref = wq.wq_matmul(d["x"], d["packed"], d["scales"], d["zeros"], p.M, p.N, p.K, p.w_bit,
                       p.group_size).cpu().numpy().astype(np.float64)
    y_oracle = oracle_y(p)
    for _ in range(2):
        out = torch.full((p.M, p.N), float("nan"), device="cuda")
        wq.wq_matmul_noalloc(d["x"], d["packed"], d["scales"], d["zeros"], p.M, p.N, p.K, p.w_bit,
                             p.group_size, out=out)
        wq.wq_check_device()
        y = out.cpu().numpy()
        assert_close(y, ref, p.K, "noalloc vs wq_matmul %s (workspace %d bytes)" % (p.name, need))
        assert_close(y, y_oracle, p.K, "noalloc vs oracle %s" % p.name)


def test_noalloc_many_token_problem_runs_one_tile_per_block():
    # a many-token problem with few tiles: with a workspace wq_matmul runs the
    # persistent stream-K kernel; without allocation, one tile per thread block
    # (no scratch).  Same result within the tolerance, bit for bit on
    # integer-exact data, and the oracle's.
    for exact in (False, True):
        p = syn.grouped("prefill noalloc", 300, 4096, 512, 4, 128, "bf16", "bf16", (0.002, 0.02), seed=9,
                        int_exact=exact)
        assert wq.wq_matmul_path(p.M, p.N, p.K, 4, 128, p.x.dtype, p.scales.dtype) == 2
        d = to_device(p)
        ref = wq.wq_matmul(d["x"], d["packed"], d["scales"], d["zeros"], p.M, p.N, p.K, 4, 128)
        out = torch.full((p.M, p.N), float("nan"), device="cuda")
        wq.wq_matmul_noalloc(d["x"], d["packed"], d["scales"], d["zeros"], p.M, p.N, p.K, 4, 128, out=out)
        wq.wq_check_device()
        if exact:
            assert torch.equal(out, ref)
        assert_close(out.cpu().numpy(), ref.cpu().numpy().astype(np.float64), p.K, "noalloc vs wq_matmul")
        rows = [0, 77, 150, 299]
        assert_close(out.cpu().numpy()[rows], oracle_y(p, rows=rows), p.K, "noalloc vs oracle")


def test_noalloc_scratch_is_used_by_a_split_problem():
    # the narrow problem splits K too finely for a cluster, so the scratch path really runs
    p = _narrow()
    assert wq.wq_workspace_bytes(p.M, p.N, p.K, p.w_bit, p.group_size) > 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    # Few column blocks over a very long K with many tokens need the most
    # scratch.  Find such a problem whose workspace exceeds the fixed array:
    # the call must return WQ_ERR_WORKSPACE and leave the output untouched.
    found = None
    for K in (65536, 131072):
        for N in (64, 128, 192, 256, 384, 512):
            for M in (64, 48, 40):
                if wq.wq_workspace_bytes(M, N, K, 4, 128) > SCRATCH_LIMIT:
                    found = (M, N, K)
                    break
            if found:
                break
        if found:
            break
    if found is None:
        pytest.skip("on this device no problem needs more than the fixed scratch")
    M, N, K = found
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    packed = torch.zeros(K * N // 2, dtype=torch.uint8, device="cuda")
    s = torch.zeros((K // 128, N), dtype=torch.bfloat16, device="cuda")
    out = torch.full((M, N), float("nan"), device="cuda")
    with pytest.raises(wq.WQError) as e:
        wq.wq_matmul_noalloc(x, packed, s, None, M, N, K, 4, 128, out=out)
    assert e.value.status == 7  # WQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool(torch.isnan(out).all())
