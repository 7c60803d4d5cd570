"""CPU oracle for weight-only quantized matmul -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs
(``cpu_baseline`` and ``--impl reference``) may import this package.  The
CUDA library never imports, links or calls it, and the two share no code.

The arithmetic lives in ``wq_oracle.c`` (plain C, fp64, k ascending); this
module only builds it with gcc and marshals numpy arrays through ctypes.
Every function's docstring names the passage it follows; see the C file for
the full statement.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile wq_oracle.c with gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared",
                               "-ffp-contract=off", "-fno-fast-math",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.wq_oracle_f16_to_f64.restype = ctypes.c_double
    lib.wq_oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.wq_oracle_bf16_to_f64.restype = ctypes.c_double
    lib.wq_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.wq_oracle_f32_to_f64.restype = ctypes.c_double
    lib.wq_oracle_f32_to_f64.argtypes = [ctypes.c_uint32]
    lib.wq_oracle_decode16_array.argtypes = [P, ctypes.c_size_t, I, P]
    lib.wq_oracle_unpack.argtypes = [P, I, I, I, P]
    lib.wq_oracle_pack.argtypes = [P, I, I, I, P]
    lib.wq_oracle_dequant.argtypes = [P, P, I, P, I, I, I, I, P]
    lib.wq_oracle_matmul_grouped.argtypes = [P, I, P, P, I, P, I, I, I, I, I, I, I, P, I, P]
    lib.wq_oracle_matmul_int8.argtypes = [P, I, P, P, I, I, I, I, I, P, I, P]
    lib.wq_oracle_t2_unpack.argtypes = [P, I, I, P]
    lib.wq_oracle_t2_pack.argtypes = [P, I, I, P]
    lib.wq_oracle_t2_matmul.argtypes = [P, P, I, I, I, P]
    for f in ("wq_oracle_decode16_array", "wq_oracle_unpack", "wq_oracle_pack",
              "wq_oracle_dequant", "wq_oracle_matmul_grouped", "wq_oracle_matmul_int8",
              "wq_oracle_t2_unpack", "wq_oracle_t2_pack", "wq_oracle_t2_matmul"):
        getattr(lib, f).restype = I
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    """Raw 16-bit patterns of an fp16/bf16 array (numpy uint16 or a torch tensor)."""
    if hasattr(a, "view") and hasattr(a, "dtype") and "torch" in type(a).__module__:
        import torch
        return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError("oracle rejected the arguments of " + what)


class Oracle:
    """The oracle's entry points, bound to one compiled copy of wq_oracle.c
    (the default build, or a deliberately mutated copy used by the pin tests)."""

    def __init__(self, lib):
        self._lib = lib

    def decode16(self, bits: np.ndarray, is_bf16: bool) -> np.ndarray:
        """fp16 / bf16 bit patterns -> fp64 values, decoded bit by bit."""
        bits = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(bits.shape, dtype=np.float64)
        _check(self._lib.wq_oracle_decode16_array(_ptr(bits), bits.size, int(is_bf16), _ptr(out)), "decode16")
        return out

    def f32_to_f64(self, bits: int) -> float:
        return self._lib.wq_oracle_f32_to_f64(int(bits) & 0xFFFFFFFF)

    def unpack(self, qw: np.ndarray, K: int, N: int, w_bit: int) -> np.ndarray:
        """Page-2 packed int32 (ceil(K/pack), N) -> uint8 codes (K, N).
        BitDistiller quant_matmul_kernel, the K loop: shift by (k % pack_num) * w_bit, mask."""
        qw = np.ascontiguousarray(qw).view(np.uint32)
        codes = np.empty((K, N), dtype=np.uint8)
        _check(self._lib.wq_oracle_unpack(_ptr(qw), K, N, w_bit, _ptr(codes)), "unpack")
        return codes

    def pack(self, codes: np.ndarray, w_bit: int) -> np.ndarray:
        """uint8 codes (K, N) -> page-2 packed int32 (ceil(K/pack), N), LSB-first along K."""
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        K, N = codes.shape
        pk = 32 // w_bit
        qw = np.empty(((K + pk - 1) // pk, N), dtype=np.uint32)
        _check(self._lib.wq_oracle_pack(_ptr(codes), K, N, w_bit, _ptr(qw)), "pack")
        return qw.view(np.int32)

    def dequant(self, qw, scales, s_is_bf16, qzeros, K, N, w_bit, group_size) -> np.ndarray:
        """fp64 (K, N) matrix of (code - zero) * scale (the reading of the cut-off
        dequant step of BitDistiller quant_matmul_kernel)."""
        qw = np.ascontiguousarray(qw).view(np.uint32)
        s = _u16(scales)
        qz = None if qzeros is None else np.ascontiguousarray(qzeros).view(np.uint32)
        w = np.empty((K, N), dtype=np.float64)
        _check(self._lib.wq_oracle_dequant(_ptr(qw), _ptr(s), int(s_is_bf16), _ptr(qz), K, N, w_bit,
                                         group_size, _ptr(w)), "dequant")
        return w

    def matmul_grouped(self, x, x_is_bf16, qw, scales, s_is_bf16, qzeros, M, N, K, w_bit, group_size,
                       n0: int = 0, n1: int | None = None, rows=None) -> np.ndarray:
        """y = x @ dequant(qw) in fp64 (BitDistiller quant_matmul_kernel, C = A x qw).
        Returns (len(rows) or M, n1 - n0)."""
        n1 = N if n1 is None else n1
        xb = _u16(x)
        qw = np.ascontiguousarray(qw).view(np.uint32)
        s = _u16(scales)
        qz = None if qzeros is None else np.ascontiguousarray(qzeros).view(np.uint32)
        r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
        nr = M if r is None else r.size
        y = np.empty((nr, n1 - n0), dtype=np.float64)
        _check(self._lib.wq_oracle_matmul_grouped(_ptr(xb), int(x_is_bf16), _ptr(qw), _ptr(s), int(s_is_bf16),
                                                _ptr(qz), M, N, K, w_bit, group_size, n0, n1,
                                                _ptr(r), nr, _ptr(y)), "matmul_grouped")
        return y

    def matmul_int8(self, x, x_is_bf16, q, scale, M, N, K, n0: int = 0, n1: int | None = None, rows=None) -> np.ndarray:
        """y = scale[n] * sum_k x[m,k] q[n,k] in fp64 (tiny-llm int8_matmul docstring)."""
        n1 = N if n1 is None else n1
        xb = _u16(x)
        if "torch" in type(q).__module__:
            q = q.detach().cpu().contiguous().numpy()
        if "torch" in type(scale).__module__:
            scale = scale.detach().cpu().contiguous().numpy()
        q = np.ascontiguousarray(q, dtype=np.int8)
        sb = np.ascontiguousarray(scale, dtype=np.float32).view(np.uint32)
        r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
        nr = M if r is None else r.size
        y = np.empty((nr, n1 - n0), dtype=np.float64)
        _check(self._lib.wq_oracle_matmul_int8(_ptr(xb), int(x_is_bf16), _ptr(q), _ptr(sb), M, N, K, n0, n1,
                                             _ptr(r), nr, _ptr(y)), "matmul_int8")
        return y

    def t2_unpack(self, packed, K: int, N: int) -> np.ndarray:
        """Liger planar 2-bit bytes (K/4, N) -> int8 weights (K, N) in {-1, 0, 1, 2}
        (Liger ops/experimental/mm_int8int2.py, unpack_weights)."""
        packed = np.ascontiguousarray(_np(packed), dtype=np.uint8)
        w = np.empty((K, N), dtype=np.int8)
        _check(self._lib.wq_oracle_t2_unpack(_ptr(packed), K, N, _ptr(w)), "t2_unpack")
        return w

    def t2_pack(self, w) -> np.ndarray:
        """int8 weights (K, N) in {-1, 0, 1, 2} -> planar bytes (K/4, N) (pack_weights)."""
        w = np.ascontiguousarray(_np(w), dtype=np.int8)
        K, N = w.shape
        packed = np.empty((K // 4, N), dtype=np.uint8)
        _check(self._lib.wq_oracle_t2_pack(_ptr(w), K, N, _ptr(packed)), "t2_pack")
        return packed

    def t2_matmul(self, x, packed, M: int, N: int, K: int) -> np.ndarray:
        """int64 y = x (M, K) int8 @ unpacked ternary weights (Liger matmul_kernel, exact)."""
        x = np.ascontiguousarray(_np(x), dtype=np.int8)
        packed = np.ascontiguousarray(_np(packed), dtype=np.uint8)
        y = np.empty((M, N), dtype=np.int64)
        _check(self._lib.wq_oracle_t2_matmul(_ptr(x), _ptr(packed), M, N, K, _ptr(y)), "t2_matmul")
        return y


def _np(a):
    if "torch" in type(a).__module__:
        return a.detach().cpu().contiguous().numpy()
    return a


def load(path: str | None = None) -> Oracle:
    """The oracle bound to the default build (path None) or to another compiled copy."""
    return Oracle(_load() if path is None else _bind(path))


_default = None


def _get() -> Oracle:
    global _default
    if _default is None:
        _default = load()
    return _default


def decode16(*a, **k): return _get().decode16(*a, **k)
def f32_to_f64(*a, **k): return _get().f32_to_f64(*a, **k)
def unpack(*a, **k): return _get().unpack(*a, **k)
def pack(*a, **k): return _get().pack(*a, **k)
def dequant(*a, **k): return _get().dequant(*a, **k)
def matmul_grouped(*a, **k): return _get().matmul_grouped(*a, **k)
def matmul_int8(*a, **k): return _get().matmul_int8(*a, **k)
def t2_unpack(*a, **k): return _get().t2_unpack(*a, **k)
def t2_pack(*a, **k): return _get().t2_pack(*a, **k)
def t2_matmul(*a, **k): return _get().t2_matmul(*a, **k)
