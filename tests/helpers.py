"""Shared helpers for the parity tests: device copies, library calls, oracle
calls (threaded over column blocks), and the tolerance of the statement of
the problem: max |y - y_oracle| <= 1e-2 * sqrt(K / 4096) * RMS(y_oracle)."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle
import weight_only_quantized_wq_gb300 as wq


def tolerance(K: int, y_ref: np.ndarray) -> float:
    rms = float(np.sqrt(np.mean(np.square(y_ref))))
    return 1e-2 * np.sqrt(K / 4096.0) * rms


def to_device(p, dev="cuda"):
    """Device copies of a synthetic problem's tensors."""
    d = {"x": p.x.to(dev), "qweight": p.qweight.to(dev), "scales": p.scales.to(dev),
         "zeros": None if p.zeros is None else p.zeros.to(dev)}
    d["packed"] = wq.wq_pack(d["qweight"], p.K, p.N, p.w_bit)
    return d


def run(p, d=None, out=None):
    d = d or to_device(p)
    return wq.wq_matmul(d["x"], d["packed"], d["scales"], d["zeros"], p.M, p.N, p.K, p.w_bit, p.group_size,
                        out=out)


def _oracle_block(p, n0, n1, rows):
    if p.w_bit == 8:
        return oracle.matmul_int8(p.x, p.x_dtype == "bf16", p.qweight, p.scales, p.M, p.N, p.K,
                                  n0=n0, n1=n1, rows=rows)
    return oracle.matmul_grouped(p.x, p.x_dtype == "bf16", p.qweight.numpy(), p.scales, p.s_dtype == "bf16",
                                 None if p.zeros is None else p.zeros.numpy(), p.M, p.N, p.K, p.w_bit,
                                 p.group_size, n0=n0, n1=n1, rows=rows)


def oracle_y(p, rows=None, threads=None) -> np.ndarray:
    """fp64 oracle output for the selected rows (all if None), computed over
    column blocks in parallel threads (the oracle's C code releases the GIL)."""
    threads = threads or min(16, os.cpu_count() or 4)
    nblk = max(1, min(threads * 2, p.N // 16))
    edges = [p.N * i // nblk for i in range(nblk + 1)]
    with cf.ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda i: _oracle_block(p, edges[i], edges[i + 1], rows), range(nblk)))
    return np.concatenate(parts, axis=1)


def assert_close(y_gpu: np.ndarray, y_ref: np.ndarray, K: int, what=""):
    tol = tolerance(K, y_ref)
    err = float(np.max(np.abs(y_gpu.astype(np.float64) - y_ref)))
    assert np.all(np.isfinite(y_gpu)), what + ": non-finite output"
    assert err <= tol, "%s: max err %.3e > tol %.3e (rms %.3e)" % (what, err, tol, tol / 1e-2 / np.sqrt(K / 4096))
    return err, tol
