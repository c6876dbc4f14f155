"""The accuracy suite on the GPU: every synthetic input of Fig. 15 and the
far-block pattern of Fig. 5, every row, for Lean P, exact P, both without
block scaling, and BF16 ("ZYFA: Speed and Accuracy of FP8 FlashAttention on
AMD CDNA4", Sec. VI, Fig. 15; Sec. IV-B2, Fig. 5).  The kernels must match
the oracle as tightly as on Gaussian inputs, so their error against fp64 is
the method's own; on the far-block pattern the kernels' error stays an order
of magnitude below the oracle's ablation in the style of the compared
kernel."""
import numpy as np
import pytest

import synthetic as S
from tests import accuracy as A
from tests import parity as P

pytestmark = pytest.mark.gpu

KINDS = list(S.FIG15_KINDS) + ["far_blocks"]
MODES = ["lean", "exact", "lean_nobs", "exact_nobs", "bf16"]
STRICT_REL_L2 = 1e-3


@pytest.fixture(scope="module")
def lib():
    import fp8_causal_flashattention_gb300 as Z
    Z.build()
    Z.load()
    return Z


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("d", [128, 192])
def test_fig15_inputs_all_rows(lib, kind, mode, d):
    N = 1024 if d == 128 else 512
    wl = S.Workload(kind, 1, 2, 1, N, d, 128, kind=kind)
    inp = S.make_inputs(wl, seed=21, fp8=mode != "bf16", bf16=mode == "bf16")
    out = P.gpu_run(inp, mode)
    rows = np.arange(wl.B * wl.Hq * wl.N)
    res = P.errors(P.gather_rows(out, wl, rows), inp, mode, rows)
    print(kind, d, mode, {k: round(v, 6) if isinstance(v, float) else v for k, v in res.items()})
    assert P.passes(res, mode), res
    assert res["rel_l2"] <= STRICT_REL_L2, res
    # the kernel's distance to fp64 is the method's own (the oracle's, with
    # the same BF16 output rounding)
    assert abs(res["rel_l2_fp64"] - res["oracle_bf16_rel_l2_fp64"]) <= \
        0.1 * res["oracle_bf16_rel_l2_fp64"] + 1e-4, res


@pytest.mark.parametrize("mode", ["lean", "exact"])
def test_far_blocks_kernel_beats_ablation(lib, mode):
    """At N = 4096 the far blocks carry enough mass that the ablation's
    output visibly shrinks; the kernel, with per-block scaling and the
    rounded row sum, stays near fp64."""
    wl = S.Workload("far_blocks", 1, 4, 1, 4096, 128, 128, kind="far_blocks")
    inp = S.make_inputs(wl, seed=22)
    out = P.gpu_run(inp, mode)
    rows = S.sample_rows(wl, per_head=128)
    got = P.gather_rows(out, wl, rows)
    import oracle
    ref, _ = oracle.attn_fp64(P.oracle_params(wl, inp, mode), inp.q8, inp.k8, inp.v8, rows)
    _, ob, _ = oracle.fwd(A.ablation_params(wl, inp), inp.q8, inp.k8, inp.v8, rows)
    ab = oracle.bf16_bits_to_f64(ob)
    e_gpu, e_ab = A.rel_rms(got, ref), A.rel_rms(ab, ref)
    print(mode, "kernel", e_gpu, "ablation", e_ab, "ablation norm",
          np.linalg.norm(ab) / np.linalg.norm(ref))
    assert e_gpu * 10 < e_ab
    assert np.linalg.norm(ab) / np.linalg.norm(ref) < 0.95
    assert abs(np.linalg.norm(got) / np.linalg.norm(ref) - 1) < 0.005
