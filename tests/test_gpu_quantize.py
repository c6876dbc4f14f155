"""GPU parity of the quantisation pass (zyfa_quantize) against the oracle.

The kernel works in FP32 and the oracle in float64.  Without smoothing or
rotation z = x / d is exact in both, so every code must match, ties included.
With a transform a kernel code may differ from the oracle's only by one step
and only where the exact value lies within the FP32 error bound ``delta``
of the midpoint between the two codes; the bound is derived below from the
arithmetic (u = 2^-24):

* mean of N values in any summation order: |err| <= gamma_N mean|x|,
  gamma_N = N u / (1 - N u), plus u |mean| for the final division;
* the transform of one row: a chain of at most 7 butterflies (D = 128) or 6
  butterflies and a 3-term DCT (D = 192), each element of the result a
  +-weighted sum of the row with weights of magnitude <= cmax = max |R|, so
  |err| <= 32 u cmax (||x - mean||_1 + ||mean err||_1), 32 covering the chain
  length, the subtraction and the constants' own rounding.

Besides the bound, differing codes must stay rare (a plausible bug moves
far more codes by far more than delta).  Codes 0x00 and 0x80 (+0 and -0)
are the same value: the sign of an exact zero after sign flips and
butterflies depends on the order of the additions, so it is not compared.
"""
import math

import numpy as np
import pytest

import synthetic as S

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module")
def lib():
    import fp8_causal_flashattention_gb300 as Z
    Z.build()
    Z.load()
    return Z


def _e4m3_values():
    import oracle
    return oracle.e4m3_decode_table()


def _inputs(shape, kind, seed):
    """BF16 bits [B, N, H, D] of a seeded tensor: 'gauss' (sigma 2.5),
    'kbias' (sigma 1 plus an N(0, 16) offset per (b, h, channel)) or
    'outlier' (4 channels per head x 20)."""
    B, N, H, D = shape
    x = S.normal(shape, seed, 20) * np.float32(2.5 if kind == "gauss" else 1.0)
    if kind == "kbias":
        x = x + S.normal((B, 1, H, D), seed, 21) * np.float32(4.0)
    elif kind == "outlier":
        rng = np.random.default_rng(seed)
        for h in range(H):
            x[:, :, h, rng.choice(D, 4, replace=False)] *= np.float32(20.0)
    return S.to_bf16_bits(x)


def _zero_sign_free(c):
    c = np.array(c, dtype=np.uint8, copy=True)
    c[c == 0x80] = 0
    return c


def _run_gpu(lib, xb, signs, smooth, static, return_mean=True):
    import torch
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    s = None if signs is None else torch.from_numpy(signs).cuda()
    res = lib.quantize(x, s, smooth=smooth, static_descale=static, return_mean=return_mean)
    torch.cuda.synchronize()
    codes = res[0].view(torch.uint8).cpu().numpy()
    d = float(res[1].cpu()[0])
    mean = res[2].cpu().numpy().astype(np.float64) if return_mean else None
    return codes, d, mean


def _mean_err_bound(xf, N):
    g = N * U / (1 - N * U)
    return g * np.mean(np.abs(xf), axis=1)                      # [B, H, D]


def _check(xb, signs, smooth, ref, codes, rows=None, mean_gpu=None):
    """Codes equal, or one step apart with z within delta of the midpoint."""
    import oracle
    from oracle import quantize as OQ
    B, N, H, D = xb.shape
    d = ref["descale"]
    xf = OQ.bf16_bits_to_f64(xb)
    if smooth:
        mu = ref["mean"]
        merr = _mean_err_bound(xf, N)
        if mean_gpu is not None:
            assert np.all(np.abs(mean_gpu - mu) <= merr + U * np.abs(mu) + 1e-300)
    flat = xf.reshape(-1, D)
    ids = np.arange(B * N * H) if rows is None else np.asarray(rows)
    bh = (ids // (N * H)) * H + ids % H
    u = flat[ids] - (ref["mean"].reshape(-1, D)[bh] if smooth else 0.0)
    merr_rows = merr.reshape(-1, D)[bh] if smooth else np.zeros_like(u)
    if signs is not None:
        cmax = float(np.max(np.abs(OQ.rotation(signs))))
        delta = 32 * U * cmax * (np.abs(u).sum(axis=1) + merr_rows.sum(axis=1))[:, None] / d
        delta = np.broadcast_to(delta, u.shape)
    elif smooth:
        delta = (2 * U * np.abs(u) + merr_rows) / d
    else:
        delta = np.zeros(u.shape)
    z = ref["z"].reshape(-1, D)
    want = _zero_sign_free(ref["codes"].reshape(-1, D))
    got = _zero_sign_free(codes.reshape(-1, D)[ids] if rows is not None else codes.reshape(-1, D))
    diff = got != want
    n_diff = int(diff.sum())
    if n_diff:
        vals = _e4m3_values()
        zg, zw = vals[got[diff]], vals[want[diff]]
        mid = 0.5 * (zg + zw)
        zz = z[diff]
        assert np.all(np.isfinite(zg)) and np.all(np.isfinite(zw)), "NaN code mismatch"
        # adjacent codes: nothing representable strictly between them
        lo, hi = np.minimum(zg, zw), np.maximum(zg, zw)
        fin = vals[np.isfinite(vals)]
        between = np.array([np.any((fin > a) & (fin < b)) for a, b in zip(lo, hi)])
        assert not between.any(), "codes more than one step apart"
        assert np.all(np.abs(zz - mid) <= delta[diff]), (
            "a differing code outside the FP32 bound",
            np.max(np.abs(zz - mid) - delta[diff]))
    assert n_diff <= max(2, 1e-4 * got.size), (n_diff, got.size)
    return n_diff


SHAPES = [
    # B, N, H, D
    (1, 1, 1, 128),
    (1, 7, 3, 128),
    (2, 100, 3, 128),
    (1, 65, 2, 192),
    (3, 64, 5, 192),
    (1, 1000, 8, 128),
    (2, 333, 4, 192),
]
MODES = [(rot, smooth, dyn) for rot in (0, 1) for smooth in (0, 1) for dyn in (1, 0)]


def _mode_id(m):
    return f"{'rot' if m[0] else 'norot'}-{'smooth' if m[1] else 'raw'}-{'dyn' if m[2] else 'static'}"


@pytest.mark.parametrize("mode", MODES, ids=[_mode_id(m) for m in MODES])
@pytest.mark.parametrize("shape", SHAPES, ids=["x".join(map(str, s)) for s in SHAPES])
def test_quantize_all_elements(lib, shape, mode):
    from oracle import quantize as OQ
    rot, smooth, dyn = mode
    kind = "kbias" if smooth else "gauss"
    xb = _inputs(shape, kind, seed=sum(shape) + 7 * rot + 3 * smooth)
    signs = S.rotation_signs(shape[3]) if rot else None
    static = None
    if not dyn:
        # a calibrated scale one binade above the per-call one
        static = 2.0 * OQ.quantize(xb, signs, bool(smooth))["descale"]
    ref = OQ.quantize(xb, signs, bool(smooth), static)
    codes, d, mean = _run_gpu(lib, xb, signs, bool(smooth), static)
    assert d == ref["descale"]
    n = _check(xb, signs, smooth, ref, codes, mean_gpu=mean if smooth else None)
    print(shape, _mode_id(mode), "differing codes:", n)


@pytest.mark.parametrize("D", [128, 192])
def test_outlier_channels_and_static_saturation(lib, D):
    """Outlier channels; a static scale 4x too small saturates at +-448."""
    from oracle import quantize as OQ
    xb = _inputs((1, 300, 4, D), "outlier", seed=31)
    signs = S.rotation_signs(D)
    for rot in (None, signs):
        small = OQ.quantize(xb, rot, False)["descale"] / 4.0
        ref = OQ.quantize(xb, rot, False, small)
        assert np.mean((ref["codes"] & 0x7F) == 0x7E) > 0.0
        codes, d, _ = _run_gpu(lib, xb, rot, False, small, return_mean=False)
        assert d == small
        _check(xb, rot, False, ref, codes)


def test_nan_inf_and_zero(lib):
    """NaN -> 0x7F, +-inf saturate; an all-zero tensor gets descale 1; the
    per-call maximum skips non-finite values."""
    from oracle import quantize as OQ
    x = np.zeros((1, 3, 2, 128), np.float32)
    xb = S.to_bf16_bits(x)
    codes, d, _ = _run_gpu(lib, xb, None, False, None, return_mean=False)
    assert d == 1.0 and not codes.any()
    x[0, 1, 0, :4] = [np.nan, np.inf, -np.inf, 3.0]
    x[0, 2, 1, 5] = -1000.0
    xb = S.to_bf16_bits(x)
    ref = OQ.quantize(xb, None, False)
    codes, d, _ = _run_gpu(lib, xb, None, False, None, return_mean=False)
    assert d == ref["descale"] == 4.0
    assert np.array_equal(codes, ref["codes"])
    assert codes[0, 1, 0, 0] == 0x7F and codes[0, 1, 0, 1] == 0x7E and codes[0, 1, 0, 2] == 0xFE
    # with rotation a NaN row stays NaN-coded and other rows are untouched
    signs = S.rotation_signs(128)
    ref = OQ.quantize(xb, signs, False, 8.0)
    codes, _, _ = _run_gpu(lib, xb, signs, False, 8.0, return_mean=False)
    assert np.all(codes[0, 1, 0] == 0x7F) and np.all(ref["codes"][0, 1, 0] == 0x7F)
    assert np.array_equal(_zero_sign_free(codes[0, 0]), _zero_sign_free(ref["codes"][0, 0]))
    assert np.array_equal(_zero_sign_free(codes[0, 2]), _zero_sign_free(ref["codes"][0, 2]))


def test_empty_tensor_writes_descale(lib):
    import torch
    Z = lib
    d = torch.full((1,), -1.0, device="cuda")
    x = torch.empty((0, 5, 2, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((0, 5, 2, 128), dtype=torch.uint8, device="cuda")
    assert Z.zyfa_quantize(x, None, 1, 0.0, out, d, None, 0, 5, 2, 128) == Z.ZYFA_OK
    assert float(d.cpu()[0]) == 1.0
    assert Z.zyfa_quantize(None, None, 0, 0.25, None, d, None, 2, 0, 2, 192) == Z.ZYFA_OK
    assert float(d.cpu()[0]) == 0.25


def test_repeat_bitwise_identical(lib):
    import torch
    xb = _inputs((2, 2000, 4, 128), "kbias", seed=5)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    s = torch.from_numpy(S.rotation_signs(128)).cuda()
    first = [t.clone() for t in lib.quantize(x, s, smooth=True, return_mean=True)]
    for _ in range(20):
        again = lib.quantize(x, s, smooth=True, return_mean=True)
        for a, b in zip(first, again):
            assert torch.equal(a.view(torch.uint8) if a.dtype == torch.float8_e4m3fn else a,
                               b.view(torch.uint8) if b.dtype == torch.float8_e4m3fn else b)


@pytest.mark.parametrize("which", ["q", "k", "v"])
def test_full_size_d128(lib, which):
    """Q, K and V of the 32-head, N = 32K, d = 128 prefill (the bench's
    quantisation step): Q rotated with a static scale, K rotated and
    smoothed with a per-call scale, V plain with a per-call scale.  The
    descale and the means cover every row; codes are compared on sampled
    rows."""
    from oracle import quantize as OQ
    wl = S.WORKLOADS["d128"]
    shape = (wl.B, wl.N, wl.Hq if which == "q" else wl.Hkv, wl.d_qk)
    xb = _inputs(shape, "kbias" if which == "k" else "gauss", seed={"q": 40, "k": 41, "v": 42}[which])
    signs = S.rotation_signs(128) if which != "v" else None
    smooth = which == "k"
    static = 2.0 ** -5 if which == "q" else None
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(shape[0] * shape[1] * shape[2], 20000, replace=False))
    rows = np.concatenate([[0], rows, [shape[0] * shape[1] * shape[2] - 1]])
    ref = OQ.quantize(xb, signs, smooth, static, rows=rows)
    codes, d, mean = _run_gpu(lib, xb, signs, smooth, static)
    assert d == ref["descale"]
    n = _check(xb, signs, smooth, ref, codes, rows=rows, mean_gpu=mean if smooth else None)
    print(which, "descale", d, "differing codes:", n, "of", rows.size * shape[3])


@pytest.mark.parametrize("D", [128, 192])
def test_quantize_then_attention_matches_oracle(lib, D):
    """The quantised, rotated Q and K go straight into the FP8 kernel with the
    device descales; the output matches the oracle's attention on the
    oracle's codes, and rotation lowers the error against fp64 attention on
    the BF16 inputs for outlier channels shared by q and k (Table XIII)."""
    import torch
    import oracle
    from oracle import quantize as OQ
    from tests import parity as P
    wl = S.Workload("qa", 1, 4, 2, 512, D, 128, kind="activation")
    q, k, v, _ = S.fp32_qkv(wl, seed=17)
    qb, kb, vb = S.to_bf16_bits(q), S.to_bf16_bits(k), S.to_bf16_bits(v)
    rows = np.arange(wl.B * wl.Hq * wl.N)
    p64 = oracle.make_params(dtype="bf16", B=wl.B, Hq=wl.Hq, Hkv=wl.Hkv, N=wl.N, d_qk=D, d_v=128)
    exact = oracle.attn_fp64(p64, qb, kb, vb, rows)[0]
    errs = {}
    for rot in (False, True):
        signs = S.rotation_signs(D) if rot else None
        st = torch.from_numpy(signs).cuda() if rot else None
        dev = [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda() for a in (qb, kb, vb)]
        q8, dq = lib.quantize(dev[0], st)
        k8, dk = lib.quantize(dev[1], st, smooth=True)
        v8, dv = lib.quantize(dev[2])
        out = lib.attention_fp8(q8, k8, v8, dq, dk, dv)
        torch.cuda.synchronize()
        got = P.gather_rows(out, wl, rows)
        rq, rk, rv = (OQ.quantize(qb, signs), OQ.quantize(kb, signs, True), OQ.quantize(vb))
        inp = S.Inputs(wl, rq["codes"], rk["codes"], rv["codes"],
                       (rq["descale"], rk["descale"], rv["descale"]))
        res = P.errors(got, inp, "lean", rows, extra=False)
        assert res["rel_l2"] <= 2e-3, res
        errs[rot] = np.linalg.norm(got - exact) / np.linalg.norm(exact)
    print("error vs fp64 on BF16 inputs: none", errs[False], "rotation", errs[True])
    assert errs[True] < 0.8 * errs[False]
