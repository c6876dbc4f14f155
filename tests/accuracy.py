"""Helpers of the accuracy suite: the error of one attention call on the
synthetic inputs of Fig. 15 and the far-block pattern of Fig. 5, for every
mode, next to an ablation of the oracle in the style of the FP8 kernel the
paper compares against ("ZYFA: Speed and Accuracy of FP8 FlashAttention on
AMD CDNA4", Sec. IV-B2 and IV-B3 with Fig. 5, Sec. VI with Fig. 15).

The ablation follows Fig. 5's description of that kernel: p rounded to e4m3
relative to the row maximum (exact exponential, no shift: sigma = 0), no
per-block scaling, and a row sum of the unrounded probabilities.  It is the
oracle with those three settings, not the other kernel itself.

Errors are relative RMS against fp64 attention on the same quantised inputs
(Sec. V-D); the P term is Sec. V-E's emulation: the exact row maximum, the
method's rounded probabilities against unrounded ones.
"""
from __future__ import annotations

import numpy as np

import oracle
import synthetic as S
from tests import parity as P

# Fig. 5's description of the compared kernel, as oracle settings
ABLATION = dict(sigma=0.0, denom_mode=oracle.DENOM_UNROUNDED)
ABLATION_MODE = "exact_nobs"


def rel_rms(x, ref) -> float:
    return float(np.linalg.norm(np.asarray(x) - ref) / np.linalg.norm(ref))


def ablation_params(wl: S.Workload, inp: S.Inputs, **extra):
    return P.oracle_params(wl, inp, ABLATION_MODE, **ABLATION, **extra)


def oracle_errors(wl: S.Workload, inp: S.Inputs, rows, modes=("lean", "exact")) -> dict:
    """Oracle-side errors against fp64 on ``rows``: each FP8 mode of the
    method and the ablation (BF16 outputs, as the kernels write)."""
    q, k, v = inp.q8, inp.k8, inp.v8
    ref, _ = oracle.attn_fp64(P.oracle_params(wl, inp, "lean"), q, k, v, rows)
    res = {}
    for m in modes:
        _, ob, _ = oracle.fwd(P.oracle_params(wl, inp, m), q, k, v, rows)
        res[m] = rel_rms(oracle.bf16_bits_to_f64(ob), ref)
    _, ob, _ = oracle.fwd(ablation_params(wl, inp), q, k, v, rows)
    res["ablation"] = rel_rms(oracle.bf16_bits_to_f64(ob), ref)
    return res


def p_term(wl: S.Workload, inp: S.Inputs, rows) -> dict:
    """Sec. V-E's P term (exact row maximum; rounded against unrounded
    probabilities, fp64 accumulation) of Lean P, exact P and the ablation,
    and each one's output norm relative to the unrounded output (below 1:
    the output shrinks)."""
    q, k, v = inp.q8, inp.k8, inp.v8
    ex = dict(max_mode=oracle.MAX_EXACT)
    pu = P.oracle_params(wl, inp, "exact", p_mode=oracle.P_UNROUNDED, **ex)
    ou, _, _ = oracle.fwd(pu, q, k, v, rows)
    res = {}
    for name, p in (("lean", P.oracle_params(wl, inp, "lean", **ex)),
                    ("exact", P.oracle_params(wl, inp, "exact", **ex)),
                    ("ablation", ablation_params(wl, inp, **ex))):
        o, _, _ = oracle.fwd(p, q, k, v, rows)
        res[name] = {"p_error": rel_rms(o, ou),
                     "norm_ratio": float(np.linalg.norm(o) / np.linalg.norm(ou))}
    return res
