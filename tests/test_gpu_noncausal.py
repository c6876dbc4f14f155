"""Non-causal attention (causal = 0: every query sees every key) against the
oracle, every mode, all rows of small ragged cases and sampled rows of a
longer one."""
import numpy as np
import pytest

import oracle
import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

CASES = [
    ("one_tile", 1, 1, 1, 128, 128),
    ("gqa", 2, 4, 2, 384, 128),
    ("mla", 1, 2, 2, 512, 192),
]


@pytest.fixture(scope="module")
def lib():
    import fp8_causal_flashattention_gb300 as Z
    Z.build()
    Z.load()
    return Z


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("mode", ["lean", "exact", "lean_nobs", "bf16"])
def test_noncausal_all_rows(lib, case, mode):
    wl = S.Workload(case[0], *case[1:], 128)
    inp = S.make_inputs(wl, seed=7, fp8=mode != "bf16", bf16=mode == "bf16")
    out = P.gpu_run(inp, mode, causal=0)
    rows = np.arange(wl.B * wl.Hq * wl.N)
    res = P.errors(P.gather_rows(out, wl, rows), inp, mode, rows, causal=0)
    print(case[0], mode, res)
    assert P.passes(res, mode), res
    assert res["rel_l2"] <= 1e-3, res


def test_noncausal_differs_from_causal(lib):
    wl = S.Workload("nc", 1, 2, 2, 256, 128, 128)
    inp = S.make_inputs(wl, seed=8)
    dev = P.to_device(inp)
    a = P.gpu_run(inp, "lean", dev, causal=0).float()
    b = P.gpu_run(inp, "lean", dev, causal=1).float()
    # the last row sees every key either way; the first row only key 0 when causal
    assert float((a[0, -1] - b[0, -1]).abs().max()) == 0.0
    assert float((a[0, 0] - b[0, 0]).abs().max()) > 0.01


def test_noncausal_long_sampled_rows(lib):
    wl = S.Workload("nc_long", 1, 4, 4, 8192, 128, 128)
    inp = S.make_inputs(wl, seed=9, bf16=True)
    rows = S.sample_rows(wl, per_head=256)
    for mode in ("lean", "exact", "bf16"):
        out = P.gpu_run(inp, mode, causal=0)
        res = P.errors(P.gather_rows(out, wl, rows), inp, mode, rows, causal=0)
        print("nc_long", mode, res)
        assert P.passes(res, mode), res
        assert res["rel_l2"] <= 1e-3, res
