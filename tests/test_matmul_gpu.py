"""wq_matmul on the GPU against the fp64 CPU oracle.

- every workload of the statement of the problem at its full size (the large
  prefill sweep on sampled rows), within max|err| <= 1e-2 sqrt(K/4096) RMS;
- integer-exact inputs (x integer in [-4, 4], scales 2^-4) where every fp32
  sum is exact in any order: the GPU must equal the oracle bit for bit;
- the symmetric path against the asymmetric one with every zero 8;
- determinism, ragged shapes, the M == 0 no-op, and canaries past the output.
"""
import numpy as np
import pytest
import torch

import weight_only_quantized_wq_gb300 as wq
from weight_only_quantized_wq_gb300 import synthetic as syn
from tests.helpers import assert_close, oracle_y, run, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make", [syn.int4_asym_tiny, syn.int8_per_channel, syn.int4_sym_decode, syn.int2_asym],
                         ids=["int4_asym_tiny", "int8_per_channel", "int4_sym_decode", "int2_asym"])
def test_workload_full_output(make):
    p = make()
    y = run(p).cpu().numpy()
    assert_close(y, oracle_y(p), p.K, p.name)


_SWEEP = {}


def _sweep():
    if "p" not in _SWEEP:
        _SWEEP["p"] = syn.int4_asym_sweep(4096)
        _SWEEP["d"] = to_device(_SWEEP["p"])
    return _SWEEP["p"], _SWEEP["d"]


@pytest.mark.parametrize("M", syn.C5_MS)
def test_prefill_sweep_sampled_rows(M):
    # every row up to 64 tokens; beyond, 64 sampled rows (first, last, random)
    full, d = _sweep()
    p = full.rows(M)
    dd = dict(d, x=d["x"][:M].contiguous())
    y = run(p, dd).cpu().numpy()
    if M <= 64:
        rows = list(range(M))
    else:
        rng = np.random.default_rng(M)
        rows = sorted(set([0, M - 1] + rng.choice(np.arange(1, M - 1), size=62, replace=False).tolist()))
        assert len(rows) == 64
    ref = oracle_y(p, rows=rows)
    assert_close(y[rows], ref, p.K, p.name)
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("M", [20, 24, 32, 40, 48, 56, 96, 128, 192])
def test_sweep_weights_mid_m_sampled_rows(M):
    # the large weights at token counts between the workloads' ones: the
    # few-token kernel with 32- and 64-row token tiles (several waves of
    # clusters), the many-token kernel with partial token tiles; called twice
    full, d = _sweep()
    p = full.rows(M)
    dd = dict(d, x=d["x"][:M].contiguous())
    for _ in range(2):
        y = run(p, dd).cpu().numpy()
        rows = sorted(set([0, M // 3, M // 2 + 1, M - 1]))
        assert_close(y[rows], oracle_y(p, rows=rows), p.K, p.name)


@pytest.mark.parametrize("M", [17, 64, 130])
def test_sweep_weights_exact_tensor_core_path(M):
    # the exact tensor-core kernel on the large weights (fp16 x with bf16
    # scales routes there at any token count above the few-token range;
    # below it the same call is checked on the few-token kernel)
    full, _ = _sweep()
    p = full.rows(M)
    p = p.__class__(**dict(p.__dict__, x=p.x.to(torch.float16), x_dtype="f16"))
    want = 0 if M <= 64 else 1
    assert wq.wq_matmul_path(M, p.N, p.K, 4, p.group_size, torch.float16, torch.bfloat16) == want
    y = run(p).cpu().numpy()
    rows = sorted(set([0, M // 2, M - 1]))
    assert_close(y[rows], oracle_y(p, rows=rows), p.K, p.name)


SHORT_K = [  # (M, K, N, group, x dtype, symmetric): below K = 4096 the bound is tighter
    (17, 512, 272, 128, "bf16", False), (65, 1024, 272, 128, "bf16", False), (256, 2048, 384, 64, "bf16", False),
    (130, 512, 144, 512, "bf16", True), (40, 1024, 128, 256, "f16", False), (256, 512, 272, 128, "f16", False),
    (300, 1024, 208, 128, "f16", True), (512, 2048, 256, 128, "f16", False), (384, 512, 512, 64, "bf16", False),
    (100, 512, 64, 64, "bf16", False), (200, 1024, 48, 1024, "bf16", True), (66, 512, 16, 128, "f16", False),
]


@pytest.mark.parametrize("M,K,N,gs,xd,sym", SHORT_K)
def test_tensor_core_paths_short_k(M, K, N, gs, xd, sym):
    # bf16 many-token problems below K = 4096 take the exact path (rounding w
    # to bf16 would not hold the bound there); fp16 ones may round w once.
    p = syn.grouped("short-k", M, K, N, 4, gs, xd, xd, (0.002, 0.02), symmetric=sym, seed=M + K + N)
    path = wq.wq_matmul_path(M, N, K, 4, gs, p.x.dtype, p.scales.dtype)
    assert path == (0 if M <= 64 else 2 if xd == "f16" else 1)
    y = run(p).cpu().numpy()
    assert_close(y, oracle_y(p), K, "short K %s" % ((M, K, N, gs, xd, sym),))


INT_EXACT = [  # (name, M, K, N, w_bit, group, x, s, symmetric)
    ("int4-asym-f16", 1, 512, 512, 4, 128, "f16", "f16", False),
    ("int4-sym-f16", 3, 4096, 1024, 4, 128, "f16", "f16", True),
    ("int2-asym-bf16", 8, 8192, 1024, 2, 64, "bf16", "bf16", False),
    ("int4-asym-bf16-M16", 16, 8192, 2048, 4, 128, "bf16", "bf16", False),
    ("int4-asym-bf16-M64", 64, 1024, 512, 4, 128, "bf16", "bf16", False),
    ("int4-perchannel-bf16", 5, 2048, 256, 4, 2048, "bf16", "bf16", False),
    ("int2-g32-f16", 2, 1024, 128, 2, 32, "f16", "bf16", False),
    ("int4-asym-bf16-M24-N400", 24, 2048, 400, 4, 64, "bf16", "bf16", False),
    ("int4-perchannel-bf16-M40", 40, 1024, 256, 4, 1024, "bf16", "bf16", False),
    ("int4-asym-f16-M52-N176", 52, 2048, 176, 4, 128, "f16", "f16", False),   # 7-octet token tile
    ("int2-asym-bf16-M21", 21, 4096, 96, 2, 64, "bf16", "bf16", False),      # 3-octet token tile
    # more tokens: the exact tensor-core path (tcgen05, group scale in fp32) ...
    ("int4-asym-bf16-M200", 200, 1024, 512, 4, 128, "bf16", "bf16", False),
    ("int4-asym-f16x-bf16s-M70", 70, 1024, 128, 4, 256, "f16", "bf16", False),
    ("int4-sym-bf16-M100-N272", 100, 2048, 272, 4, 64, "bf16", "bf16", True),
    # ... and the many-token one (weight rounded once: exact here, scale 2^-4)
    ("int4-sym-f16-M128", 128, 2048, 256, 4, 64, "f16", "f16", True),
    ("int4-asym-f16-M300-N272", 300, 512, 272, 4, 512, "f16", "f16", False),
    ("int4-asym-bf16-M256-K4096", 256, 4096, 256, 4, 128, "bf16", "bf16", False),
]


INT_EXACT_PATH = {"int4-asym-bf16-M200": 1, "int4-asym-f16x-bf16s-M70": 1, "int4-sym-bf16-M100-N272": 1,
                  "int4-sym-f16-M128": 2, "int4-asym-f16-M300-N272": 2, "int4-asym-bf16-M256-K4096": 2}


@pytest.mark.parametrize("case", INT_EXACT, ids=[c[0] for c in INT_EXACT])
def test_integer_exact_bitwise(case):
    name, M, K, N, wb, gs, xd, sd, sym = case
    dt = {"f16": torch.float16, "bf16": torch.bfloat16}
    assert wq.wq_matmul_path(M, N, K, wb, gs, dt[xd], dt[sd]) == INT_EXACT_PATH.get(name, 0)
    p = syn.grouped(name, M, K, N, wb, gs, xd, sd, (0, 0), symmetric=sym, seed=11, int_exact=True)
    y = run(p).cpu().numpy().astype(np.float64)
    ref = oracle_y(p)
    assert np.array_equal(y, ref), "max diff %g" % np.max(np.abs(y - ref))


ONE_TILE_RAGGED = [  # (M, K, N, x dtype, integer-exact): many tiles (one per CTA), token and channel tails
    (300, 4096, 10000, "bf16", False),   # 2 x 40 tiles; the last channel block holds 16 channels
    (1000, 4096, 6160, "f16", False),    # 4 x 25 tiles
    (520, 4096, 9744, "bf16", True),     # 3 x 39 tiles, integer-exact: bit for bit
]


@pytest.mark.parametrize("M,K,N,xd,exact", ONE_TILE_RAGGED)
def test_prefill_one_tile_ragged(M, K, N, xd, exact):
    # the many-token one-tile kernel (x ring and weight ring of their own) with
    # partial token tiles and partial channel blocks, on sampled rows
    p = syn.grouped("one-tile", M, K, N, 4, 128, xd, xd, (0.002, 0.02), seed=M + N, int_exact=exact)
    assert wq.wq_matmul_path(M, N, K, 4, 128, p.x.dtype, p.scales.dtype) == 2
    assert wq.wq_workspace_bytes(M, N, K, 4, 128) == 0  # enough tiles: one per CTA, no stream-K
    y = run(p).cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(M)
    rows = sorted(set([0, 255, 256, M - 1] + rng.choice(np.arange(M), size=12, replace=False).tolist()))
    ref = oracle_y(p, rows=rows)
    if exact:
        assert np.array_equal(y[rows], ref), "max diff %g" % np.max(np.abs(y[rows] - ref))
    else:
        assert_close(y[rows], ref, K, p.name)


TWO_TERM = [  # (M, K, N, integer-exact): bf16 below K = 4096 on grids of >= 128 tiles (path 3)
    (1024, 2048, 4096, False),   # 4 x 32 tiles of 256 tokens x 128 channels
    (1024, 2048, 4096, True),    # integer-exact: bit for bit
    (300, 1024, 16400, False),   # 2 x 129 tiles, a 16-channel last block, a partial token tile
]


@pytest.mark.parametrize("M,K,N,exact", TWO_TERM)
def test_two_term_weights(M, K, N, exact):
    # each weight enters the MMA as its bf16 rounding plus the bf16 rounding of
    # the residue: within 2^-16 of the weight, far inside the bound at any K
    p = syn.grouped("two-term", M, K, N, 4, 128, "bf16", "bf16", (0.002, 0.02), seed=M + N, int_exact=exact)
    assert wq.wq_matmul_path(M, N, K, 4, 128, p.x.dtype, p.scales.dtype) == 3
    y = run(p).cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(M + N)
    rows = sorted(set([0, 255, 256, M - 1] + rng.choice(np.arange(M), size=12, replace=False).tolist()))
    ref = oracle_y(p, rows=rows)
    if exact:
        assert np.array_equal(y[rows], ref), "max diff %g" % np.max(np.abs(y[rows] - ref))
    else:
        err, tol = assert_close(y[rows], ref, K, p.name)
        assert err <= 0.05 * tol, "two-term weights should sit far inside the bound (%g of it)" % (err / tol)


def test_int8_integer_exact_bitwise():
    p = syn.int8("int8-exact", 16, 4096, 1024, "bf16", (0.001, 0.01), seed=12, int_exact=True)
    y = run(p).cpu().numpy().astype(np.float64)
    ref = oracle_y(p)
    # the sum is exact; one fp32 multiply by the scale, correctly rounded
    assert np.array_equal(y, ref.astype(np.float32).astype(np.float64))


def test_symmetric_equals_zero8():
    p = syn.int4_sym_decode()
    d = to_device(p)
    ys = run(p, d)
    G = p.K // p.group_size
    z8 = torch.full(((G + 7) // 8, p.N), 0x88888888 - 2 ** 32, dtype=torch.int32, device="cuda")
    ya = wq.wq_matmul(d["x"], d["packed"], d["scales"], z8, p.M, p.N, p.K, 4, p.group_size)
    assert torch.equal(ys, ya)


def test_deterministic():
    for make in (syn.int4_sym_decode, syn.int2_asym, syn.int8_per_channel):
        p = make()
        d = to_device(p)
        assert torch.equal(run(p, d), run(p, d))


RAGGED = [  # (M, K, N, w_bit, group) -- tails of token tiles, CTA column blocks, splits, groups
    (3, 256, 80, 4, 64), (13, 512, 48, 4, 128), (17, 1024, 272, 2, 64), (33, 512, 208, 4, 32),
    (7, 4096, 16, 4, 128), (2, 8192, 32, 2, 128), (40, 640, 96, 8, 640), (1, 32, 16, 8, 32), (9, 64, 16, 4, 16),
    # M > 16 on the exact tensor-core path: partial token tiles and 128-channel blocks
    (65, 4096, 64, 4, 256), (100, 4096, 144, 4, 128), (17, 64, 16, 4, 64), (33, 192, 48, 4, 64),
    # M > 64 without a tensor-core path (group 32, int2): 64-row slices of the few-token kernel
    (130, 256, 48, 4, 32), (200, 1024, 64, 2, 64),
]


@pytest.mark.parametrize("M,K,N,wb,gs", RAGGED)
def test_ragged_shapes(M, K, N, wb, gs):
    if wb == 8:
        p = syn.int8("int8-ragged", M, K, N, "bf16", (0.001, 0.01), seed=M + K)
    else:
        p = syn.grouped("ragged", M, K, N, wb, gs, "bf16" if M % 2 else "f16", "bf16", (0.005, 0.02),
                        seed=M + K + N)
    y = run(p).cpu().numpy()
    assert_close(y, oracle_y(p), K, "ragged %s" % ((M, K, N, wb, gs),))


LONG_K = [  # (M, K, N, w_bit, group, x dtype): K = 65536, the most the ternary path accepts
    (1, 65536, 32, 4, 16, "bf16"),     # 4096 groups: many K splits, partials through the workspace
    (5, 65536, 48, 2, 64, "f16"),
    (3, 65536, 16, 8, 65536, "bf16"),  # int8 per channel
    (300, 65536, 512, 4, 128, "bf16"), # many-token kernel: 1024 stages per tile
]


@pytest.mark.parametrize("M,K,N,wb,gs,xd", LONG_K)
def test_long_k(M, K, N, wb, gs, xd):
    if wb == 8:
        p = syn.int8("int8-long-k", M, K, N, xd, (0.001, 0.01), seed=K + N)
    else:
        p = syn.grouped("long-k", M, K, N, wb, gs, xd, xd, (0.002, 0.02), seed=K + N + M)
    y = run(p).cpu().numpy()
    rows = sorted(set([0, M // 2, M - 1]))
    assert_close(y[rows], oracle_y(p, rows=rows), K, "long K %s" % ((M, K, N, wb, gs),))
    wq.wq_check_device()


def test_zero_rows_is_noop_and_canaries():
    p = syn.int4_asym_tiny()
    d = to_device(p)
    out = torch.full((p.N + 64,), float("nan"), device="cuda")
    wq.wq_matmul(d["x"], d["packed"], d["scales"], d["zeros"], 0, p.N, p.K, 4, 128, out=out)
    torch.cuda.synchronize()
    assert torch.isnan(out).all()
    # one row written, the guard band after it untouched
    sentinel = -12345.0
    buf = torch.full((p.N + 64,), sentinel, device="cuda")
    wq.wq_matmul(d["x"], d["packed"], d["scales"], d["zeros"], 1, p.N, p.K, 4, 128, out=buf)
    torch.cuda.synchronize()
    assert bool((buf[p.N:] == sentinel).all())
    assert not bool((buf[:p.N] == sentinel).any())
    wq.wq_check_device()


def test_workspace_too_small_is_rejected():
    # one column block over a long K: more K splits than one cluster reduces,
    # so the partial sums need the caller's workspace
    p = syn.grouped("int4-asym narrow", 4, 8192, 64, 4, 128, "bf16", "bf16", (0.002, 0.02), seed=5)
    need = wq.wq_workspace_bytes(p.M, p.N, p.K, 4, p.group_size)
    assert need > 0
    d = to_device(p)
    small = torch.zeros(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(wq.WQError) as e:
        wq.wq_matmul(d["x"], d["packed"], d["scales"], d["zeros"], p.M, p.N, p.K, 4, p.group_size, workspace=small)
    assert e.value.status == 7
    # with enough workspace the same call matches the oracle
    y = run(p, d).cpu().numpy()
    assert_close(y, oracle_y(p), p.K, p.name)


def test_cluster_split_needs_no_workspace():
    # few column blocks over a long K: the K splits are reduced inside a
    # thread-block cluster, so no workspace is needed, and the result matches
    p = syn.grouped("int4-asym cluster split", 8, 8192, 2048, 4, 128, "bf16", "bf16", (0.002, 0.02), seed=6)
    assert wq.wq_workspace_bytes(p.M, p.N, p.K, 4, p.group_size) == 0
    d = to_device(p)
    y = run(p, d).cpu().numpy()
    assert_close(y, oracle_y(p), p.K, p.name)


PERSIST = [  # (M, K, N, x dtype): few tiles, so persistent CTAs with stream-K shares
    (256, 4096, 256, "bf16"),    # one tile, two CTAs
    (300, 4096, 1024, "bf16"),   # 8 tiles (two token tiles), 16 CTAs
    (1024, 4096, 1024, "f16"),   # 16 tiles, 32 CTAs
    (700, 8192, 2304, "bf16"),   # 27 tiles, 54 CTAs: shares cut tiles at odd stages
    (130, 1024, 128, "f16"),     # one 128-token tile (one accumulator), 16 stages
]


@pytest.mark.parametrize("M,K,N,xd", PERSIST)
def test_prefill_persistent_shares_match_one_tile_per_cta(M, K, N, xd):
    # the many-token kernel with a workspace runs persistent (stream-K shares,
    # cut tiles finished by a fix-up); without one, one tile per CTA.  Both
    # must match the oracle, and each other bit for bit on integer-exact data.
    for exact in (False, True):
        p = syn.grouped("persist", M, K, N, 4, 128, xd, xd, (0.002, 0.02), seed=M + N, int_exact=exact)
        assert wq.wq_matmul_path(M, N, K, 4, 128, p.x.dtype, p.scales.dtype) == 2
        d = to_device(p)
        need = wq.wq_workspace_bytes(M, N, K, 4, 128)
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        y_sk = wq.wq_matmul(d["x"], d["packed"], d["scales"], d["zeros"], M, N, K, 4, 128, workspace=ws)
        y_sk2 = wq.wq_matmul(d["x"], d["packed"], d["scales"], d["zeros"], M, N, K, 4, 128, workspace=ws)
        tiny = torch.zeros(16, dtype=torch.uint8, device="cuda")
        y_dp = wq.wq_matmul(d["x"], d["packed"], d["scales"], d["zeros"], M, N, K, 4, 128, workspace=tiny)
        wq.wq_check_device()
        assert need > 16384  # the persistent kernel has its partial tiles
        assert torch.equal(y_sk, y_sk2)  # deterministic
        assert int(ws[:16384].count_nonzero()) == 0  # flags back at zero
        if exact:
            assert torch.equal(y_sk, y_dp)
        rows = sorted(set([0, M - 1] + np.random.default_rng(M).choice(M, size=min(M, 30), replace=False).tolist()))
        ref = oracle_y(p, rows=rows)
        for y in (y_sk, y_dp):
            yy = y.cpu().numpy()[rows]
            if exact:
                assert np.array_equal(yy.astype(np.float64), ref)
            else:
                assert_close(yy, ref, K, "persistent %s" % ((M, K, N, xd),))
