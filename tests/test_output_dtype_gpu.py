"""wq_matmul_ex: fp16 / bf16 output.  The kernels accumulate in fp32 exactly
as for the fp32 output and round once, to nearest even, on store, so the
16-bit output must equal torch's round-to-nearest-even cast of wq_matmul's
fp32 output bit for bit, on every kernel path; and it must stay within the
accepted error of the fp64 oracle plus the output's own rounding."""
import numpy as np
import pytest
import torch

import weight_only_quantized_wq_gb300 as wq
from weight_only_quantized_wq_gb300 import synthetic as syn
from tests.helpers import oracle_y, tolerance, to_device

pytestmark = pytest.mark.gpu

CASES = {  # name -> problem; the comment gives the kernel path
    "decode-int4-M16": lambda: syn.grouped("d16", 16, 4096, 2048, 4, 128, "bf16", "bf16", (0.002, 0.02), seed=21),
    "decode-int2-M8": lambda: syn.grouped("d8", 8, 2048, 512, 2, 64, "bf16", "bf16", (0.01, 0.05), seed=22),
    "decode-int8-M16": lambda: syn.int8("i8", 16, 2048, 1024, "bf16", (0.001, 0.01), seed=23),
    "decode-workspace-split": lambda: syn.grouped("ws", 4, 8192, 64, 4, 128, "bf16", "bf16", (0.002, 0.02), seed=5),
    "decode-64-row-slices": lambda: syn.grouped("sl", 100, 1024, 272, 4, 32, "f16", "f16", (0.002, 0.02), seed=24),
    "exact-tc-M100": lambda: syn.grouped("tc", 100, 2048, 400, 4, 128, "bf16", "bf16", (0.002, 0.02), seed=25),
    "prefill-M300": lambda: syn.grouped("pf", 300, 4096, 272, 4, 128, "bf16", "bf16", (0.002, 0.02), seed=26),
    "two-term-M129": lambda: syn.grouped("tt", 129, 512, 16384, 4, 128, "bf16", "bf16", (0.002, 0.02), seed=27),
}
PATH = {"exact-tc-M100": 1, "prefill-M300": 2, "two-term-M129": 3}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("odt", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_16bit_output_is_the_rounded_fp32_result(name, odt):
    p = CASES[name]()
    d = to_device(p)
    assert wq.wq_matmul_path(p.M, p.N, p.K, p.w_bit, p.group_size, p.x.dtype, p.scales.dtype) == PATH.get(name, 0)
    y32 = wq.wq_matmul(d["x"], d["packed"], d["scales"], d["zeros"], p.M, p.N, p.K, p.w_bit, p.group_size)
    # a guard band after the 16-bit output must stay untouched
    buf = torch.full((p.M * p.N + 64,), -7.0, dtype=odt, device="cuda")
    out = buf[:p.M * p.N].view(p.M, p.N)
    wq.wq_matmul_ex(d["x"], d["packed"], d["scales"], d["zeros"], p.M, p.N, p.K, p.w_bit, p.group_size,
                    out=out, out_dtype=odt)
    wq.wq_check_device()
    assert torch.equal(out, y32.to(odt)), "16-bit output differs from the rounded fp32 result"
    assert bool((buf[p.M * p.N:] == -7.0).all())
    ref = oracle_y(p)
    y = out.float().cpu().numpy().astype(np.float64)
    u = 2.0 ** -11 if odt == torch.float16 else 2.0 ** -8
    bound = tolerance(p.K, ref) + u * np.abs(ref)
    assert np.all(np.abs(y - ref) <= bound)


def test_bad_output_dtype_is_rejected():
    p = CASES["decode-int4-M16"]()
    d = to_device(p)
    out = torch.empty((p.M, p.N), dtype=torch.float16, device="cuda")
    st = wq.binding.lib().wq_matmul_ex(d["x"].data_ptr(), wq.binding.WQ_BF16, d["packed"].data_ptr(),
                                       d["scales"].data_ptr(), wq.binding.WQ_BF16, d["zeros"].data_ptr(),
                                       p.M, p.N, p.K, 4, 128, out.data_ptr(), 7, None, 0, None)
    assert st == wq.binding.STATUS.index("WQ_ERR_DTYPE")
