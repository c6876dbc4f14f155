"""The failure path without a GPU fault: a bounded wait that nothing
satisfies runs out, the kernel returns, zyfa_last_device_status() reports
ZYFA_ERR_TIMEOUT once, and the context keeps working."""
import time

import numpy as np
import pytest

import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_is_reported_and_context_survives():
    import torch
    import fp8_causal_flashattention_gb300 as Z
    Z.build()
    Z.load()
    assert Z.zyfa_last_device_status() == Z.ZYFA_OK          # clear any earlier state
    t0 = time.time()
    assert Z.zyfa_selftest_timeout() == Z.ZYFA_OK
    assert Z.zyfa_last_device_status() == Z.ZYFA_ERR_TIMEOUT
    assert 1.0 < time.time() - t0 < 30.0                    # the 1.5 s budget, bounded
    assert Z.zyfa_last_device_status() == Z.ZYFA_OK          # reported once, then cleared
    wl = S.Workload("after", 1, 2, 2, 256, 128, 128)
    inp = S.make_inputs(wl, seed=12)
    out = P.gpu_run(inp, "lean")
    torch.cuda.synchronize()
    assert Z.zyfa_last_device_status() == Z.ZYFA_OK
    rows = np.arange(wl.B * wl.Hq * wl.N)
    res = P.errors(P.gather_rows(out, wl, rows), inp, "lean", rows, extra=False)
    assert res["rel_l2"] <= 1e-3
