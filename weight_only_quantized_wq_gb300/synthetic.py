"""Seeded synthetic inputs for the weight-only quantized matmul workloads.

This module only draws random numbers; it holds none of the method's
arithmetic (no packing, no dequantization, no matmul).  Packed weights and
packed zeros are drawn directly as uniform random 32-bit words: every bit
pattern of a page-2 word is a valid packing, and uniform random bits give
codes that are uniform over [0, 2^w_bit - 1] in every field.  Unused fields
of the last packed-zeros row hold random bits too; both the library and the
oracle must ignore them.

Draw order for every problem: x, weights, scales, zeros -- one
``torch.Generator('cpu')`` seeded per problem.  The same tensors feed the
CUDA library (after a copy to the device) and the CPU oracle.
"""
from __future__ import annotations

import dataclasses

import torch

F16, BF16, F32 = "f16", "bf16", "f32"
_TORCH = {F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32}


@dataclasses.dataclass
class Problem:
    name: str
    M: int
    K: int
    N: int
    w_bit: int              # 2, 4 (grouped, page-2 layout) or 8 (int8 per-channel)
    group_size: int         # along K; == K for per-channel
    x_dtype: str
    s_dtype: str
    x: torch.Tensor         # (M, K)
    qweight: torch.Tensor   # int32 (K/pack, N) for w_bit 2/4; int8 (N, K) for w_bit 8
    scales: torch.Tensor    # (K/group_size, N) f16/bf16; (N,) f32 for w_bit 8
    zeros: torch.Tensor | None  # int32 (ceil(G/pack), N) or None (symmetric)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.K * self.N

    def weight_bytes(self) -> int:
        """Packed weights + scales + packed zeros, each counted once."""
        b = self.qweight.numel() * self.qweight.element_size() + self.scales.numel() * self.scales.element_size()
        if self.zeros is not None:
            b += self.zeros.numel() * 4
        return b

    def total_bytes(self) -> int:
        """Algorithmic bytes of one matmul: weights + scales + zeros + x + fp32 y."""
        return self.weight_bytes() + self.x.numel() * self.x.element_size() + self.M * self.N * 4

    def rows(self, m: int) -> "Problem":
        """The same weights with only the first m activation rows."""
        return dataclasses.replace(self, M=m, x=self.x[:m].contiguous(), name=f"{self.name}[M={m}]")


def _words(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randint(-(2 ** 31), 2 ** 31, shape, generator=gen, dtype=torch.int64).to(torch.int32)


def _uniform(gen, shape, lo, hi, dtype) -> torch.Tensor:
    return (torch.rand(shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo).to(_TORCH[dtype])


def grouped(name, M, K, N, w_bit, group_size, x_dtype, s_dtype, s_range, symmetric=False,
            seed=0, int_exact=False) -> Problem:
    """Page-2 grouped problem: x ~ N(0,1), uniform random packed words, scales
    uniform in s_range, uniform random packed zero words (None if symmetric).
    int_exact: x integer in [-4, 4] and every scale 2^-4 (all terms exact)."""
    gen = torch.Generator("cpu").manual_seed(seed)
    pack = 32 // w_bit
    G = K // group_size
    if int_exact:
        x = torch.randint(-4, 5, (M, K), generator=gen).to(_TORCH[x_dtype])
    else:
        x = torch.randn((M, K), generator=gen, dtype=torch.float32).to(_TORCH[x_dtype])
    qw = _words(gen, ((K + pack - 1) // pack, N))
    if int_exact:
        s = torch.full((G, N), 2.0 ** -4, dtype=_TORCH[s_dtype])
    else:
        s = _uniform(gen, (G, N), s_range[0], s_range[1], s_dtype)
    z = None if symmetric else _words(gen, ((G + pack - 1) // pack, N))
    return Problem(name, M, K, N, w_bit, group_size, x_dtype, s_dtype, x, qw, s, z)


def int8(name, M, K, N, x_dtype, s_range, seed=0, int_exact=False) -> Problem:
    """tiny-llm int8 problem: x ~ N(0,1), q (N, K) int8 uniform in [-127, 127],
    fp32 per-output-channel scale uniform in s_range."""
    gen = torch.Generator("cpu").manual_seed(seed)
    if int_exact:
        x = torch.randint(-4, 5, (M, K), generator=gen).to(_TORCH[x_dtype])
    else:
        x = torch.randn((M, K), generator=gen, dtype=torch.float32).to(_TORCH[x_dtype])
    q = torch.randint(-127, 128, (N, K), generator=gen, dtype=torch.int64).to(torch.int8)
    s = _uniform(gen, (N,), s_range[0], s_range[1], F32)
    return Problem(name, M, K, N, 8, K, x_dtype, F32, x, q, s, None)


@dataclasses.dataclass
class TernaryProblem:
    """Liger planar ternary problem: x (M, K) int8, packed (K/4, N) uint8."""
    name: str
    M: int
    K: int
    N: int
    x: torch.Tensor
    packed: torch.Tensor

    @property
    def flops(self) -> int:
        return 2 * self.M * self.K * self.N

    def weight_bytes(self) -> int:
        return self.packed.numel()

    def total_bytes(self) -> int:
        """Algorithmic bytes: packed weights + int8 x + int32 y, each once."""
        return self.packed.numel() + self.x.numel() + self.M * self.N * 4


# bytes whose four 2-bit fields are all below 3 (weights -1, 0, 1 stored plus one)
_TERNARY_BYTES = torch.tensor([b for b in range(256) if all((b >> (2 * i)) & 3 != 3 for i in range(4))],
                              dtype=torch.uint8)


def ternary(name, M, K, N, seed=0, all_fields=False) -> TernaryProblem:
    """x uniform int8 in [-128, 127]; each packed byte uniform over the bytes
    whose fields are all 0..2 (ternary weights), or over all 256 bytes
    (all_fields: field 3, weight 2, included)."""
    gen = torch.Generator("cpu").manual_seed(seed)
    x = torch.randint(-128, 128, (M, K), generator=gen, dtype=torch.int64).to(torch.int8)
    if all_fields:
        packed = torch.randint(0, 256, (K // 4, N), generator=gen, dtype=torch.int64).to(torch.uint8)
    else:
        idx = torch.randint(0, len(_TERNARY_BYTES), (K // 4, N), generator=gen, dtype=torch.int64)
        packed = _TERNARY_BYTES[idx]
    return TernaryProblem(name, M, K, N, x, packed)


def ternary_decode(seed=0):
    """Ternary int2 (BitNet-style) decode: M=16, K=8192, N=8192."""
    return ternary("ternary-int2 M16 K8192 N8192", 16, 8192, 8192, seed=seed)


# The five workloads, with the sizes and distributions of the statement of the problem.
def int4_asym_tiny(seed=0):
    """int4 asymmetric, group 128: M=1, K=512, N=512, fp16 x and scales."""
    return grouped("int4-asym-g128 M1 K512 N512", 1, 512, 512, 4, 128, F16, F16, (0.005, 0.02), seed=seed)


def int8_per_channel(seed=0):
    """int8 per-output-channel: M=16, K=4096, N=4096, bf16 x, fp32 scale."""
    return int8("int8-perchannel M16 K4096 N4096", 16, 4096, 4096, BF16, (0.001, 0.01), seed=seed)


def int4_sym_decode(seed=0):
    """int4 symmetric (zero 8), group 128: M=1, K=4096, N=11008, fp16."""
    return grouped("int4-sym-g128 M1 K4096 N11008", 1, 4096, 11008, 4, 128, F16, F16, (0.002, 0.02),
                   symmetric=True, seed=seed)


def int2_asym(seed=0):
    """int2 asymmetric, group 64: M=8, K=8192, N=8192, bf16."""
    return grouped("int2-asym-g64 M8 K8192 N8192", 8, 8192, 8192, 2, 64, BF16, BF16, (0.01, 0.05), seed=seed)


C5_MS = (16, 64, 256, 1024, 4096)


def int4_asym_sweep(M=4096, seed=0):
    """int4 asymmetric, group 128, K=8192, N=28672, bf16; x drawn for M=4096,
    smaller M take its first rows."""
    p = grouped("int4-asym-g128 K8192 N28672", 4096, 8192, 28672, 4, 128, BF16, BF16, (0.002, 0.02), seed=seed)
    return p.rows(M)


def int4_asym_short_k(M=128, seed=0):
    """int4 asymmetric, group 128, K=2048, N=28672, bf16: a shorter K than the
    sweep, where the many-token kernel's rounding of w to bf16 would not hold
    the accepted error, so more than 64 tokens run on the exact path."""
    return grouped("int4-asym-g128 K2048 N28672 M%d" % M, M, 2048, 28672, 4, 128, BF16, BF16, (0.002, 0.02),
                   seed=seed)


WORKLOADS = {
    "int4_asym_tiny": int4_asym_tiny,
    "int8_per_channel": int8_per_channel,
    "int4_sym_decode": int4_sym_decode,
    "int2_asym": int2_asym,
    "int4_asym_sweep": int4_asym_sweep,
    "int4_asym_short_k": int4_asym_short_k,
    "ternary_decode": ternary_decode,
}
