"""wq_matmul_noalloc: the entry point for callers that cannot allocate device
memory (it uses a fixed scratch array inside the library instead of a caller
workspace).  Its output must match wq_matmul's, within the tolerance the
other parity tests use, on two calls in a row (the second call reuses the
scratch the first one left behind).  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import weight_only_quantized_wq_gb300 as wq
from weight_only_quantized_wq_gb300 import synthetic as syn
from tests.helpers import assert_close, to_device

pytestmark = pytest.mark.gpu


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
    for _ in range(2):
        out = torch.full((p.M, p.N), float("nan"), device="cuda")
        wq.wq_matmul_noalloc(d["x"], d["packed"], d["scales"], d["zeros"], p.M, p.N, p.K, p.w_bit,
                             p.group_size, out=out)
        wq.wq_check_device()
        assert_close(out.cpu().numpy(), ref, p.K, "noalloc %s (workspace %d bytes)" % (p.name, need))


def test_noalloc_scratch_is_used_by_a_split_problem():
    # the narrow problem splits K too finely for a cluster, so the scratch path really runs
    p = _narrow()
    assert wq.wq_workspace_bytes(p.M, p.N, p.K, p.w_bit, p.group_size) > 0
