"""The accuracy suite's CPU side: Fig. 15's synthetic inputs match their
descriptions, and the oracle reproduces Fig. 5's effect -- without per-block
scaling and with the row sum of unrounded probabilities, probabilities of
blocks far below the maximum are lost from the numerator only, so the
output shrinks and the P error grows along the row; per-block scaling with
the rounded row sum keeps it near the rounding error of p ("ZYFA: Speed and
Accuracy of FP8 FlashAttention on AMD CDNA4", Sec. IV-B2, IV-B3, Fig. 5,
Fig. 15)."""
import numpy as np
import pytest

import synthetic as S
from tests import accuracy as A

N = 1024


def _logits(kind, N=N, d=128, Hq=2, Hkv=1):
    wl = S.Workload(kind, 1, Hq, Hkv, N, d, 128, kind=kind)
    q, k, v, _ = S.fp32_qkv(wl, seed=0)
    L = np.einsum("nd,md->nm", q[0, :, 0].astype(np.float64),
                  k[0, :, 0].astype(np.float64)) / np.sqrt(d)
    return wl, q, k, v, L


def _causal(L):
    return L[np.tril_indices(L.shape[0])]


@pytest.mark.parametrize("kind,sd", [("logit_sd1", 1.0), ("logit_sd4", 4.0),
                                     ("logit_sd16", 16.0)])
def test_logit_sd(kind, sd):
    _, _, _, _, L = _logits(kind)
    assert abs(np.std(_causal(L)) / sd - 1) < 0.03


def test_gaussian_sigma():
    _, q, k, v, _ = _logits("f15_gaussian")
    for x in (q, k, v):
        assert abs(np.std(x) / S.F15_SIGMA - 1) < 0.02


def test_stepped_max():
    _, _, _, _, L = _logits("stepped_max")
    last = L[N - 1]                                  # sees every key
    bmax = last.reshape(-1, 64).max(axis=1)
    base = _logits("logit_sd1")[4][N - 1].reshape(-1, 64).max(axis=1)
    # each block is F15_STEP_NATS above the previous one, on top of N(0,1)
    # logits (up to one channel's share of them)
    steps = np.diff(bmax - base)
    assert np.all(np.abs(steps - S.F15_STEP_NATS) < 0.7)
    assert np.all(np.diff(np.maximum.accumulate(bmax)) >= 0)
    assert bmax[-1] - bmax[0] > 0.8 * S.F15_STEP_NATS * (N // 64 - 1)


def test_sink4():
    _, _, k, _, _ = _logits("sink4")
    _, _, k0, _, _ = _logits("logit_sd1")
    assert np.array_equal(k[:, :4], k0[:, :4] * np.float32(8.0))
    assert np.array_equal(k[:, 4:], k0[:, 4:])


@pytest.mark.parametrize("kind", ["rising", "alternating"])
def test_ramp(kind):
    _, _, _, _, L = _logits(kind)
    _, _, _, _, L0 = _logits("logit_sd1")
    D = L - L0                                       # the added ramp (plus channel 0's change)
    j = np.arange(N)
    for i in (N - 1, N - 2):
        slope = np.polyfit(j, D[i], 1)[0] * N
        ramp = kind == "rising" or i % 2 == 0
        if ramp:
            assert abs(slope / S.F15_RAMP_NATS - 1) < 0.05, (i, slope)
        else:
            assert abs(slope) < 0.05 * S.F15_RAMP_NATS, (i, slope)


def test_sink_flat():
    _, _, _, _, L = _logits("sink_flat")
    rest = L[:, 1:][np.tril_indices(N - 1)]          # keys 1..i of rows 1..N-1
    assert abs(np.std(rest) / S.F15_FLAT_SD - 1) < 0.1
    gap = L[1:, 0] - np.array([L[i, 1:i + 1].mean() for i in range(1, N)])
    assert abs(np.mean(gap) - S.F15_SINK_NATS) < 0.1


def test_full_range():
    _, q, k, v, _ = _logits("full_range")
    for x in (q, k, v):
        e = np.log2(np.abs(x.astype(np.float64)))
        lo, hi = S.F15_RANGE
        assert e.min() >= lo and e.max() <= hi
        # uniform in [lo, hi]: quantiles on the line
        qs = np.quantile(e, [0.1, 0.5, 0.9])
        assert np.all(np.abs(qs - (lo + (hi - lo) * np.array([0.1, 0.5, 0.9]))) < 0.1)
        assert abs(np.mean(x > 0) - 0.5) < 0.01


def test_far_blocks_is_sink_with_offset_values():
    wl = S.Workload("fb", 1, 2, 1, N, 128, 128, kind="far_blocks")
    q, k, v, meta = S.fp32_qkv(wl)
    wl0 = S.Workload("s", 1, 2, 1, N, 128, 128, kind="sink")
    q0, k0, v0, _ = S.fp32_qkv(wl0)
    assert np.array_equal(q, q0) and np.array_equal(k, k0)
    assert np.array_equal(v, v0 + np.float32(S.FAR_BLOCKS_V_MEAN))


def test_fig5_effect_in_oracle():
    """Fig. 5: the compared kernel's settings lose the far blocks from the
    numerator only, so the output shrinks and the P error grows with the row
    length; the method's per-block scaling and rounded row sum keep the P
    error near that of rounding p (Sec. IV-B2: 11% against 1.0% on one
    layer of a real model)."""
    res = {}
    for n in (1024, 2048):
        wl = S.Workload("fb", 1, 4, 1, n, 128, 128, kind="far_blocks")
        inp = S.make_inputs(wl)
        res[n] = A.p_term(wl, inp, S.sample_rows(wl, per_head=128))
    print(res)
    ab, lean, exact = res[2048]["ablation"], res[2048]["lean"], res[2048]["exact"]
    assert ab["p_error"] > 0.05 and ab["norm_ratio"] < 0.97
    assert res[2048]["ablation"]["p_error"] > 1.5 * res[1024]["ablation"]["p_error"]
    assert lean["p_error"] < 0.005 and abs(lean["norm_ratio"] - 1) < 0.002
    assert exact["p_error"] < 0.001 and abs(exact["norm_ratio"] - 1) < 0.001
    assert ab["p_error"] > 10 * lean["p_error"]


def test_ablation_settings_each_matter():
    """Per-block scaling is the change that keeps the far blocks: alone (with
    the unrounded row sum) it brings the P error below 1% and keeps the
    output's norm; the rounded row sum alone keeps the weights summing to one
    but moves the far blocks' mass onto the near ones, so its P error stays
    large.  Both together are at least as good as block scaling alone."""
    import oracle
    from tests import parity as P
    wl = S.Workload("fb", 1, 4, 1, 2048, 128, 128, kind="far_blocks")
    inp = S.make_inputs(wl)
    rows = S.sample_rows(wl, per_head=128)
    ex = dict(max_mode=oracle.MAX_EXACT)
    q, k, v = inp.q8, inp.k8, inp.v8
    ou, _, _ = oracle.fwd(P.oracle_params(wl, inp, "exact", p_mode=oracle.P_UNROUNDED, **ex),
                          q, k, v, rows)
    n_u = np.linalg.norm(ou)
    o_bs, _, _ = oracle.fwd(A.ablation_params(wl, inp, block_scale=1, **ex), q, k, v, rows)
    o_rs, _, _ = oracle.fwd(P.oracle_params(wl, inp, "exact_nobs", sigma=0.0, **ex),
                            q, k, v, rows)
    o_m, _, _ = oracle.fwd(P.oracle_params(wl, inp, "exact", sigma=0.0, **ex), q, k, v, rows)
    e_bs, e_rs, e_m = (A.rel_rms(o, ou) for o in (o_bs, o_rs, o_m))
    print("block scale only", e_bs, "rounded sum only", e_rs, "both", e_m)
    assert abs(np.linalg.norm(o_bs) / n_u - 1) < 0.005
    assert np.linalg.norm(o_rs) / n_u > 1.0          # no shrinkage, mass moved instead
    assert e_rs > 0.01
    assert e_bs < 0.01 and e_m <= e_bs and e_m < 0.1 * e_rs
