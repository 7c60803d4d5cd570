"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin takes an ``oracle.Oracle`` and raises AssertionError when it
disagrees with a hand-worked value (tests/golden/pins.json), a library
routine (numpy integer matmul, torch dtype casts), a closed form, or an
invariant.  The same pins run against deliberately broken copies of the
oracle (test_oracle_mutants.py) to show that each plausible mistake fails
at least one of them.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "pins.json")


def _hexwords(lst, rows, cols):
    return np.array([int(h, 16) for h in lst], dtype=np.uint32).reshape(rows, cols).view(np.int32)


def _f16(vals):
    return np.array(vals, dtype=np.float16).view(np.uint16)


def pin_golden(orc):
    """Hand-worked values for unpacking, zeros, and tiny matmuls."""
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        if c.get("t2"):
            packed = np.array(c["packed"], dtype=np.uint8).reshape(c["K"] // 4, c["N"])
            w = orc.t2_unpack(packed, c["K"], c["N"])
            assert w.ravel().tolist() == c["w"], (c["id"], w)
            assert np.array_equal(orc.t2_pack(w), packed), c["id"]
            x = np.array(c["x"], dtype=np.int8).reshape(c["M"], c["K"])
            y = orc.t2_matmul(x, packed, c["M"], c["N"], c["K"])
            assert y.ravel().tolist() == c["y"], (c["id"], y)
        elif "codes" in c:
            pk = 32 // c["w_bit"]
            qw = _hexwords(c["qweight_hex"], (c["K"] + pk - 1) // pk, c["N"])
            got = orc.unpack(qw, c["K"], c["N"], c["w_bit"]).ravel().tolist()
            assert got == c["codes"], (c["id"], got)
            back = orc.pack(np.array(c["codes"], dtype=np.uint8).reshape(c["K"], c["N"]), c["w_bit"])
            assert np.array_equal(back.view(np.uint32), qw.view(np.uint32)), c["id"]
        elif "zeros" in c:
            # zeros packed along groups: probe group g with one-hot x and unit scales
            G, N, wb = c["G"], c["N"], c["w_bit"]
            pk = 32 // wb
            K = G * pk  # one packed weight row per group, all codes 0
            qw = np.zeros((K // pk, N), dtype=np.int32)
            qz = _hexwords(c["qzeros_hex"], (G + pk - 1) // pk, N)
            s = _f16(np.ones((G, N)))
            for g in range(G):
                x = np.zeros((1, K), dtype=np.float16)
                x[0, g * pk] = 1.0
                y = orc.matmul_grouped(x.view(np.uint16), False, qw, s, False, qz, 1, N, K, wb, pk)
                assert y[0, 0] == -c["zeros"][g], (c["id"], g, y)
        elif "q" in c:
            y = orc.matmul_int8(_f16(c["x"]).reshape(1, -1), False, np.array(c["q"], dtype=np.int8),
                                np.array(c["scale"], dtype=np.float32), c["M"], c["N"], c["K"])
            assert y.ravel().tolist() == c["y"], (c["id"], y)
        else:
            pk = 32 // c["w_bit"]
            G = c["K"] // c["group_size"]
            qw = _hexwords(c["qweight_hex"], (c["K"] + pk - 1) // pk, c["N"])
            qz = None if c["qzeros_hex"] is None else _hexwords(c["qzeros_hex"], (G + pk - 1) // pk, c["N"])
            s = _f16(c["scales"]).reshape(G, c["N"])
            x = _f16(c["x"]).reshape(c["M"], c["K"])
            y = orc.matmul_grouped(x, False, qw, s, False, qz, c["M"], c["N"], c["K"], c["w_bit"], c["group_size"])
            assert y.ravel().tolist() == c["y"], (c["id"], y)


def pin_decoders(orc):
    """All 65536 fp16 and bf16 bit patterns against torch's own casts."""
    pats = np.arange(65536, dtype=np.uint16)
    t = torch.from_numpy(pats.view(np.int16).copy())
    for is_bf16, dt in ((False, torch.float16), (True, torch.bfloat16)):
        ref = t.view(dt).to(torch.float64).numpy()
        got = orc.decode16(pats, is_bf16)
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], ref[~nan]), is_bf16
    rng = np.random.default_rng(1)
    bits = np.concatenate([rng.integers(0, 2 ** 32, 4000, dtype=np.uint64).astype(np.uint32),
                           np.array([0, 1, 0x80000000, 0x7f7fffff, 0x00800000, 0x3f800000], dtype=np.uint32)])
    ref = bits.view(np.float32).astype(np.float64)
    for b, r in zip(bits, ref):
        g = orc.f32_to_f64(int(b))
        assert (np.isnan(g) and np.isnan(r)) or g == r, hex(int(b))


def pin_pack_identity(orc):
    """unpack(pack(codes)) == codes (ragged K too) and pack(unpack(W)) == W."""
    rng = np.random.default_rng(2)
    for wb in (2, 4, 8):
        pk = 32 // wb
        for K, N in ((pk, 1), (3 * pk, 5), (5 * pk + 3, 7), (64, 33)):
            codes = rng.integers(0, 2 ** wb, (K, N), dtype=np.uint8)
            qw = orc.pack(codes, wb)
            assert qw.shape == ((K + pk - 1) // pk, N)
            assert np.array_equal(orc.unpack(qw, K, N, wb), codes), (wb, K, N)
        K, N = 4 * pk, 9
        words = rng.integers(0, 2 ** 32, (K // pk, N), dtype=np.uint64).astype(np.uint32)
        words[0, :3] = [0, 0xFFFFFFFF, 0x80000000]
        codes = orc.unpack(words.view(np.int32), K, N, wb)
        assert np.array_equal(orc.pack(codes, wb).view(np.uint32), words), wb


def pin_numpy_integer_matmul(orc):
    """group_size = K, zeros 0, scale 1, integer x: the oracle equals numpy's
    int64 x @ codes (a library routine), on a non-square problem."""
    rng = np.random.default_rng(3)
    for wb, (M, K, N) in ((4, (3, 64, 5)), (2, (2, 96, 7))):
        pk = 32 // wb
        codes = rng.integers(0, 2 ** wb, (K, N), dtype=np.uint8)
        xi = rng.integers(-4, 5, (M, K))
        qz = np.zeros((1, N), dtype=np.int32)
        s = _f16(np.ones((1, N)))
        y = orc.matmul_grouped(_f16(xi), False, orc.pack(codes, wb), s, False, qz, M, N, K, wb, K)
        assert np.array_equal(y, (xi.astype(np.int64) @ codes.astype(np.int64)).astype(np.float64)), wb


def pin_grouped_closed_form(orc):
    """Groups with distinct power-of-two scales s[g, n] = 2^-(g + n % 3) and
    per-(group, column) zeros: y * 2^(G+1) is the integer
    sum over groups of 2^(G+1-g-n%3) * (x_g @ (Q_g - Z_g)), computed with numpy
    int64 matmuls from the codes and zeros the test drew."""
    rng = np.random.default_rng(4)
    for wb, (M, K, N, gs), xbf in ((4, (4, 128, 6, 32), False), (2, (3, 192, 5, 64), True), (4, (2, 96, 3, 16), True)):
        pk = 32 // wb
        G = K // gs
        codes = rng.integers(0, 2 ** wb, (K, N), dtype=np.uint8)
        zeros = rng.integers(0, 2 ** wb, (G, N), dtype=np.uint8)
        xi = rng.integers(-4, 5, (M, K))
        sc = np.array([[2.0 ** -(g + n % 3) for n in range(N)] for g in range(G)])
        xb = (torch.tensor(xi, dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16) if xbf
              else _f16(xi))
        sb = torch.tensor(sc, dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        y = orc.matmul_grouped(xb, xbf, orc.pack(codes, wb), sb, True, orc.pack(zeros, wb), M, N, K, wb, gs)
        acc = np.zeros((M, N), dtype=np.int64)
        for g in range(G):
            d = codes[g * gs:(g + 1) * gs].astype(np.int64) - zeros[g].astype(np.int64)[None, :]
            colw = np.array([2 ** (G + 1 - g - n % 3) for n in range(N)], dtype=np.int64)
            acc += colw[None, :] * (xi[:, g * gs:(g + 1) * gs].astype(np.int64) @ d)
        assert np.array_equal(y * 2.0 ** (G + 1), acc.astype(np.float64)), (wb, M, K, N, gs)


def pin_symmetric_equals_zero8(orc):
    """Symmetric int4 (NULL zeros) equals the asymmetric path with every zero 8
    (packed words 0x88888888); symmetric int2 equals zeros 2 (0xAAAAAAAA)."""
    rng = np.random.default_rng(5)
    for wb, word in ((4, 0x88888888), (2, 0xAAAAAAAA)):
        M, K, N, gs = 2, 128, 4, 64
        pk = 32 // wb
        G = K // gs
        qw = rng.integers(0, 2 ** 32, (K // pk, N), dtype=np.uint64).astype(np.uint32).view(np.int32)
        x = _f16(rng.standard_normal((M, K)))
        s = _f16(rng.uniform(0.01, 0.02, (G, N)))
        qz = np.full(((G + pk - 1) // pk, N), word, dtype=np.uint32).view(np.int32)
        a = orc.matmul_grouped(x, False, qw, s, False, None, M, N, K, wb, gs)
        b = orc.matmul_grouped(x, False, qw, s, False, qz, M, N, K, wb, gs)
        assert np.array_equal(a, b), wb


def pin_int8_numpy(orc):
    """int8 per-channel: integer x, power-of-two scales -> numpy int64 (x @ q.T) * scale exactly."""
    rng = np.random.default_rng(6)
    M, K, N = 3, 40, 6
    xi = rng.integers(-4, 5, (M, K))
    q = rng.integers(-128, 128, (N, K)).astype(np.int8)
    sc = np.array([2.0 ** -(n % 4) for n in range(N)], dtype=np.float32)
    xb = torch.tensor(xi, dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = orc.matmul_int8(xb, True, q, sc, M, N, K)
    ref = (xi.astype(np.int64) @ q.astype(np.int64).T).astype(np.float64) * sc.astype(np.float64)[None, :]
    assert np.array_equal(y, ref)


def pin_slicing(orc):
    """Row and column selection return the matching block of the full result."""
    rng = np.random.default_rng(7)
    M, K, N, wb, gs = 5, 64, 12, 4, 32
    qw = rng.integers(0, 2 ** 32, (K // 8, N), dtype=np.uint64).astype(np.uint32).view(np.int32)
    qz = rng.integers(0, 2 ** 32, (1, N), dtype=np.uint64).astype(np.uint32).view(np.int32)
    x = _f16(rng.standard_normal((M, K)))
    s = _f16(rng.uniform(0.01, 0.02, (K // gs, N)))
    full = orc.matmul_grouped(x, False, qw, s, False, qz, M, N, K, wb, gs)
    part = orc.matmul_grouped(x, False, qw, s, False, qz, M, N, K, wb, gs, n0=3, n1=9, rows=[4, 0])
    assert np.array_equal(part, full[[4, 0], 3:9])
    q8 = rng.integers(-127, 128, (N, K)).astype(np.int8)
    s8 = rng.uniform(0.001, 0.01, N).astype(np.float32)
    f8 = orc.matmul_int8(x, False, q8, s8, M, N, K)
    p8 = orc.matmul_int8(x, False, q8, s8, M, N, K, n0=2, n1=11, rows=[1, 3])
    assert np.array_equal(p8, f8[[1, 3], 2:11])


def _pack_np(codes, wb):
    """Page-layout packing written out with numpy shifts (independent of the
    oracle's packer): field k % pack of word [k // pack][n], LSB first."""
    K, N = codes.shape
    pk = 32 // wb
    words = np.zeros(((K + pk - 1) // pk, N), dtype=np.uint64)
    for k in range(K):
        words[k // pk] |= codes[k].astype(np.uint64) << np.uint64(wb * (k % pk))
    return words.astype(np.uint32).view(np.int32)


def pin_dequant_closed_form(orc):
    """dequant(qw, s, qz)[k, n] == (code - zero[g, n]) * scale[g, n], g = k // group_size,
    computed with numpy from the codes, zeros and scales the test drew (scales
    widened by torch's own cast); symmetric (no qzeros) uses zero 2^(w_bit - 1).
    One-hot rows of x through matmul_grouped give the same rows exactly."""
    rng = np.random.default_rng(8)
    for wb, (K, N, gs), sbf in ((4, (96, 5, 32), True), (2, (128, 3, 64), False), (4, (64, 4, 64), False)):
        G = K // gs
        codes = rng.integers(0, 2 ** wb, (K, N), dtype=np.uint8)
        zeros = rng.integers(0, 2 ** wb, (G, N), dtype=np.uint8)
        sc = torch.tensor(rng.uniform(0.003, 3.0, (G, N)), dtype=torch.bfloat16 if sbf else torch.float16)
        s64 = sc.to(torch.float64).numpy()
        sbits = sc.view(torch.int16).numpy().view(np.uint16)
        qw = _pack_np(codes, wb)
        for qz, z in ((_pack_np(zeros, wb), zeros.astype(np.float64)),
                      (None, np.full((G, N), 2.0 ** (wb - 1)))):
            got = orc.dequant(qw, sbits, sbf, qz, K, N, wb, gs)
            gi = np.arange(K) // gs
            ref = (codes.astype(np.float64) - z[gi]) * s64[gi]
            assert np.array_equal(got, ref), (wb, K, N, gs, qz is None)
            for k in (0, gs - 1, K - 1):
                x = np.zeros((1, K), dtype=np.float16)
                x[0, k] = 1.0
                y = orc.matmul_grouped(x.view(np.uint16), False, qw, sbits, sbf, qz, 1, N, K, wb, gs)
                assert np.array_equal(y[0], got[k]), (wb, k)


def pin_t2_numpy(orc):
    """Ternary planar int2: bytes built with numpy shifts from weights the test
    drew (plane k // R in bits 2 (k // R), row k % R) unpack to those weights;
    the matmul equals numpy's int64 x @ w; pack and unpack are inverse (also on
    random bytes, whose field 3 stands for 2)."""
    rng = np.random.default_rng(9)
    for K, N, M in ((8, 3, 2), (64, 5, 3), (256, 7, 4)):
        R = K // 4
        w = rng.integers(-1, 2, (K, N)).astype(np.int8)
        packed = np.zeros((R, N), dtype=np.uint8)
        for k in range(K):
            packed[k % R] |= ((w[k] + 1).astype(np.uint8) << np.uint8(2 * (k // R)))
        assert np.array_equal(orc.t2_unpack(packed, K, N), w), K
        x = rng.integers(-128, 128, (M, K)).astype(np.int8)
        ref = x.astype(np.int64) @ w.astype(np.int64)
        assert np.array_equal(orc.t2_matmul(x, packed, M, N, K), ref), K
        assert np.array_equal(orc.t2_pack(w), packed), K
        raw = rng.integers(0, 256, (R, N)).astype(np.uint8)
        assert np.array_equal(orc.t2_pack(orc.t2_unpack(raw, K, N)), raw), K
    # extremes: every weight 2 (field 3) and x = -128 over K = 4096: -128 * 2 * 4096
    K = 4096
    packed = np.full((K // 4, 2), 0xFF, dtype=np.uint8)
    x = np.full((1, K), -128, dtype=np.int8)
    assert orc.t2_matmul(x, packed, 1, 2, K).tolist() == [[-1048576, -1048576]]


ALL_PINS = [pin_golden, pin_decoders, pin_pack_identity, pin_numpy_integer_matmul,
            pin_grouped_closed_form, pin_symmetric_equals_zero8, pin_int8_numpy, pin_slicing,
            pin_dequant_closed_form, pin_t2_numpy]
