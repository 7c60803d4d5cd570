"""wq_pack / wq_unpack on the GPU: bit-exact against the oracle's unpacking
of the page layout (and q^T bytes for int8), at every workload's shape."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_quantized_wq_gb300 as wq
from weight_only_quantized_wq_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

SHAPES = [  # (K, N, w_bit)
    (512, 512, 4), (4096, 11008, 4), (8192, 28672, 4), (8192, 8192, 2), (4096, 4096, 8),
    (64, 16, 4), (128, 48, 2), (32, 16, 8), (192, 80, 4),
]


@pytest.mark.parametrize("K,N,w_bit", SHAPES)
def test_pack_unpack_bitexact(K, N, w_bit):
    gen = torch.Generator("cpu").manual_seed(K * 7 + N + w_bit)
    if w_bit == 8:
        q = torch.randint(-128, 128, (N, K), generator=gen, dtype=torch.int64).to(torch.int8)
        ref = q.numpy().T.view(np.uint8)
    else:
        q = torch.randint(-(2 ** 31), 2 ** 31, (K * w_bit // 32, N), generator=gen, dtype=torch.int64).to(torch.int32)
        q[0, :3] = torch.tensor([0, -1, -(2 ** 31)], dtype=torch.int32)  # 0, 0xFFFFFFFF, 0x80000000
        ref = oracle.unpack(q.numpy(), K, N, w_bit)
    qd = q.cuda()
    packed = wq.wq_pack(qd, K, N, w_bit)
    assert packed.numel() == K * N * w_bit // 8
    codes = wq.wq_unpack(packed, K, N, w_bit).cpu().numpy()
    assert np.array_equal(codes, ref)
    # the repack is a permutation of bits: total popcount is preserved
    pin = np.unpackbits(q.numpy().view(np.uint8)).sum()
    pout = np.unpackbits(packed.cpu().numpy()).sum()
    assert pin == pout
    # deterministic
    assert torch.equal(wq.wq_pack(qd, K, N, w_bit), packed)


def test_pack_does_not_write_past_output():
    K, N, w = 128, 32, 4
    q = torch.randint(-(2 ** 31), 2 ** 31, (K // 8, N), dtype=torch.int64).to(torch.int32).cuda()
    buf = torch.full((K * N // 2 + 256,), 0xA5, dtype=torch.uint8, device="cuda")
    wq.wq_pack(q, K, N, w, packed_out=buf)
    torch.cuda.synchronize()
    assert bool((buf[K * N // 2:] == 0xA5).all())
