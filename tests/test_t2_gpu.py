"""Ternary int2 (Liger ops/experimental/mm_int8int2.py) on the GPU against the
oracle: the repack is bit-exact (the tiled layout unpacks to the planar
fields), and the int32 product equals the oracle's exact int64 sum bit for
bit, over token counts that take one kernel launch or 64-row slices, ragged
column blocks, long K split over clusters or through the workspace, field 3
(weight 2) included, and the extreme sum 2^24 at K = 65536."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_wq_gb300 as wq
from weight_only_quantized_wq_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _run(p):
    packed = wq.wq_t2_pack(p.packed.cuda(), p.K, p.N)
    y = wq.wq_t2_matmul(p.x.cuda(), packed, p.M, p.N, p.K)
    wq.wq_check_device()
    return packed, y.cpu().numpy()


SHAPES = [  # (M, K, N, all_fields)
    (1, 4096, 4096, False), (16, 8192, 1024, False), (8, 2048, 512, True), (64, 1024, 272, False),
    (3, 128, 16, True), (100, 1024, 48, False), (33, 512, 208, True), (4, 16384, 64, False),
]


@pytest.mark.parametrize("M,K,N,full", SHAPES)
def test_t2_matmul_bitexact(M, K, N, full):
    p = syn.ternary("t2", M, K, N, seed=M + K + N, all_fields=full)
    packed, y = _run(p)
    codes = wq.wq_unpack(packed, K, N, 2).cpu().numpy().astype(np.int16)
    assert np.array_equal(codes - 1, oracle.t2_unpack(p.packed, K, N))
    ref = oracle.t2_matmul(p.x, p.packed, M, N, K)
    assert y.dtype == np.int32
    assert np.array_equal(y.astype(np.int64), ref)


def test_t2_decode_workload_and_determinism():
    p = syn.ternary_decode()
    packed = wq.wq_t2_pack(p.packed.cuda(), p.K, p.N)
    x = p.x.cuda()
    y1 = wq.wq_t2_matmul(x, packed, p.M, p.N, p.K)
    y2 = wq.wq_t2_matmul(x, packed, p.M, p.N, p.K)
    assert torch.equal(y1, y2)
    ref = oracle.t2_matmul(p.x, p.packed, p.M, p.N, p.K)
    assert np.array_equal(y1.cpu().numpy().astype(np.int64), ref)


def test_t2_extreme_sum_is_exact():
    # every field 3 (weight 2) and x = -128 over K = 65536: -2^24, still exact
    M, K, N = 2, 65536, 32
    packed_h = torch.full((K // 4, N), 0xFF, dtype=torch.uint8)
    x_h = torch.full((M, K), -128, dtype=torch.int8)
    x_h[1, ::2] = 127
    p = syn.TernaryProblem("t2-extreme", M, K, N, x_h, packed_h)
    _, y = _run(p)
    ref = oracle.t2_matmul(x_h, packed_h, M, N, K)
    assert ref[0, 0] == -(1 << 24)
    assert np.array_equal(y.astype(np.int64), ref)


def test_t2_workspace_too_small_is_rejected():
    p = syn.ternary("t2", 16, 1024, 256, seed=3)
    packed = wq.wq_t2_pack(p.packed.cuda(), p.K, p.N)
    need = wq.wq_t2_workspace_bytes(p.M, p.N, p.K)
    assert need >= p.M * p.K * 2
    small = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(wq.WQError) as e:
        wq.wq_t2_matmul(p.x.cuda(), packed, p.M, p.N, p.K, workspace=small)
    assert e.value.status == 7


def test_t2_shared_workspace_across_shapes():
    # one workspace for calls of several shapes, some splitting K through its
    # counters and partial sums, some not: each must match the oracle
    shapes = [(4, 16384, 64), (16, 16384, 64), (4, 16384, 128), (1, 16384, 64), (64, 1024, 272), (4, 16384, 256)]
    need = max(wq.wq_t2_workspace_bytes(M, N, K) for (M, K, N) in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for i, (M, K, N) in enumerate(shapes):
        p = syn.ternary("t2", M, K, N, seed=100 + i)
        packed = wq.wq_t2_pack(p.packed.cuda(), K, N)
        y = wq.wq_t2_matmul(p.x.cuda(), packed, M, N, K, workspace=ws).cpu().numpy().astype(np.int64)
        assert np.array_equal(y, oracle.t2_matmul(p.x, p.packed, M, N, K)), (M, K, N)
