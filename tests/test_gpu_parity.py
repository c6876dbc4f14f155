"""GPU parity of the CUDA path against the CPU oracle, small and ragged cases
(every row checked).  Calls the library through its C ABI binding."""
import numpy as np
import pytest

import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

FP8_MODES = ["lean", "exact", "lean_nobs", "exact_nobs"]

SMALL = [
    # name, B, Hq, Hkv, N, d_qk
    ("one_tile", 1, 1, 1, 128, 128),
    ("pr1", 1, 1, 1, 256, 128),
    ("gqa_batch", 2, 4, 2, 384, 128),
    ("mqa", 1, 3, 1, 640, 128),
    ("long_few_heads", 1, 2, 2, 1024, 128),
    ("mla_small", 1, 2, 2, 384, 192),
    ("mla_gqa", 2, 4, 1, 256, 192),
]


@pytest.fixture(scope="module")
def lib():
    import fp8_causal_flashattention_gb300 as Z
    Z.build()
    Z.load()
    return Z


def _wl(name, B, Hq, Hkv, N, d):
    return S.Workload(name, B, Hq, Hkv, N, d, 128)


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
@pytest.mark.parametrize("mode", FP8_MODES + ["bf16"])
def test_small_all_rows(lib, case, mode):
    wl = _wl(*case)
    inp = S.make_inputs(wl, seed=3, fp8=mode != "bf16", bf16=mode == "bf16")
    out = P.gpu_run(inp, mode)
    rows = np.arange(wl.B * wl.Hq * wl.N)
    res = P.errors(P.gather_rows(out, wl, rows), inp, mode, rows)
    print(case[0], mode, res)
    assert P.passes(res, mode), res


def test_pr1_workload_matches_oracle(lib):
    """B=1, H=1, N=256, d=128, seed 0: all rows, Lean P and exact P."""
    wl = S.WORKLOADS["pr1"]
    inp = S.make_inputs(wl, bf16=True)
    rows = np.arange(wl.N)
    for mode in ("lean", "exact", "bf16"):
        res = P.errors(P.gather_rows(P.gpu_run(inp, mode), wl, rows), inp, mode, rows)
        print("pr1", mode, res)
        assert P.passes(res, mode), (mode, res)


def test_repeat_launches_bitwise_identical(lib):
    import torch
    wl = _wl("rep", 1, 4, 2, 1024, 128)
    inp = S.make_inputs(wl, seed=5)
    dev = P.to_device(inp)
    first = P.gpu_run(inp, "lean", dev).clone()
    for _ in range(50):
        assert torch.equal(P.gpu_run(inp, "lean", dev), first)


def test_device_status_clean_after_runs(lib):
    import fp8_causal_flashattention_gb300 as Z
    wl = _wl("st", 1, 2, 2, 512, 128)
    inp = S.make_inputs(wl, seed=6)
    P.gpu_run(inp, "exact")
    assert Z.zyfa_last_device_status() == Z.ZYFA_OK
