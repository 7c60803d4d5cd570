"""The failure path of the library's bounded barrier waits, without any GPU
fault: through the test hook of include/wq_testing.h the few-token kernel
runs with a short wait limit while its producers withhold one ring stage, so
the consumers' wait for it runs out.  The kernel must return (no hang),
wq_check_device must report WQ_ERR_TIMEOUT once and clear it, and the next
normal call on the same device must match the oracle."""
import pytest

import weight_only_quantized_wq_gb300 as wq
from weight_only_quantized_wq_gb300 import synthetic as syn
from tests.helpers import assert_close, oracle_y, run, to_device

pytestmark = pytest.mark.gpu

CASES = {  # name -> (problem, stage withheld); one launch each, K split as the planner chooses
    "one-split-middle-stage": (lambda: syn.int4_sym_decode(), 1),
    "one-split-first-stage": (lambda: syn.int4_sym_decode(), 0),
    "cluster-split": (lambda: syn.grouped("cl", 8, 8192, 2048, 4, 128, "bf16", "bf16", (0.002, 0.02), seed=6), 0),
    "workspace-split": (lambda: syn.grouped("ws", 4, 8192, 64, 4, 128, "bf16", "bf16", (0.002, 0.02), seed=5), 0),
    "int8": (lambda: syn.int8("i8", 16, 4096, 1024, "bf16", (0.001, 0.01), seed=7), 0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_wait_runs_out_reports_timeout_and_device_recovers(name):
    make, stage = CASES[name]
    p = make()
    d = to_device(p)
    wq.wq_check_device()  # nothing pending
    wq.binding.wq_testing_decode_timeout(d["x"], d["packed"], d["scales"], d["zeros"], p.M, p.N, p.K, p.w_bit,
                                         p.group_size, wait_limit_cycles=200000, withhold_stage=stage)
    with pytest.raises(wq.WQError) as e:
        wq.wq_check_device()
    assert e.value.status == wq.binding.STATUS.index("WQ_ERR_TIMEOUT")
    wq.wq_check_device()  # the status word was cleared
    y = run(p, d).cpu().numpy()
    wq.wq_check_device()
    assert_close(y, oracle_y(p), p.K, "after a timeout: " + name)
