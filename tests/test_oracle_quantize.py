"""Pins of the quantisation-pass oracle (CPU only).

Each test checks oracle/quantize.py against something other than itself:
SciPy's Hadamard matrix and DCT, a butterfly Walsh-Hadamard transform written
here, orthogonality and the softmax invariances that Sec. V-A states,
footnote 25's factor of 128, the closed form of the power-of-two descale,
PyTorch's e4m3 cast, and the direction of Table XIII.
"""
import math

import numpy as np
import pytest
import scipy.fft
import scipy.linalg
import torch

import synthetic as S
from oracle import quantize as OQ
from tests import brute_force as bf


def _fwht(a):
    """Unnormalised Walsh-Hadamard transform over the last axis, by
    butterflies (x + y, x - y) on index pairs (j, j + h)."""
    a = np.array(a, dtype=np.float64)
    n = a.shape[-1]
    h = 1
    while h < n:
        v = a.reshape(*a.shape[:-1], n // (2 * h), 2, h)
        x, y = v[..., 0, :].copy(), v[..., 1, :].copy()
        v[..., 0, :] = x + y
        v[..., 1, :] = x - y
        a = v.reshape(*a.shape[:-1], n)
        h *= 2
    return a


def _bf16(shape, seed, scale=1.0):
    x = S.normal(shape, seed, 7) * np.float32(scale)
    return S.to_bf16_bits(x)


def test_hadamard_is_scipy_sylvester():
    for n in [1, 2, 4, 8, 16, 32, 64, 128, 256]:
        ref = scipy.linalg.hadamard(n) / math.sqrt(n)
        assert np.allclose(OQ.hadamard(n), ref, rtol=0, atol=1e-15)


def test_dct2_is_scipy_orthonormal_dct():
    for m in range(1, 9):
        ref = scipy.fft.dct(np.eye(m), type=2, norm="ortho", axis=0)
        assert np.allclose(OQ.dct2(m), ref, rtol=0, atol=1e-14)


def test_odd_part():
    """Sec. V-A: m = 1 for D = 128 and m = 3 for D = 192."""
    assert OQ.odd_part(128) == 1 and OQ.odd_part(192) == 3
    assert OQ.odd_part(64) == 1 and OQ.odd_part(96) == 3


def test_rotation_d128_is_signed_fwht():
    s = S.rotation_signs(128)
    x = S.normal((50, 128), 1, 8).astype(np.float64)
    ref = _fwht(x * s) / math.sqrt(128.0)
    assert np.allclose(x @ OQ.rotation(s), ref, rtol=0, atol=1e-12)


def test_rotation_d192_is_inverse_dct_of_fwht():
    """y = x R with R = diag(s)(C_3 kron H_64): the 3 x 64 view of x*s is
    Hadamard-transformed along its rows, then C_3^T (the inverse of the
    orthonormal DCT-II) mixes the three rows."""
    s = S.rotation_signs(192)
    x = S.normal((40, 192), 2, 8).astype(np.float64)
    t = _fwht((x * s).reshape(40, 3, 64)) / 8.0
    ref = scipy.fft.idct(t, type=2, norm="ortho", axis=1).reshape(40, 192)
    assert np.allclose(x @ OQ.rotation(s), ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("D", [64, 128, 192, 256])
def test_rotation_orthogonal_scores_unchanged(D):
    """Sec. V-A: R is orthogonal, so (QR)(KR)^T = QK^T."""
    R = OQ.rotation(S.rotation_signs(D, seed=3))
    assert np.allclose(R @ R.T, np.eye(D), rtol=0, atol=1e-13)
    q = S.normal((20, D), 4, 8).astype(np.float64)
    k = S.normal((30, D), 5, 8).astype(np.float64)
    assert np.allclose((q @ R) @ (k @ R).T, q @ k.T, rtol=0, atol=1e-11)


def test_rotation_rejects_non_signs():
    with pytest.raises(ValueError):
        OQ.rotation(np.array([1.0, 0.5, -1.0, 1.0]))


def test_footnote25_one_shared_channel_factor(golden):
    """All energy of q and k in one shared channel: the rotation lowers
    sum_i q_i^2 k_i^2 by a factor of D = 128 (footnote 25)."""
    g = golden["rotation_one_channel_factor"]
    D = g["D"]
    R = OQ.rotation(S.rotation_signs(D))
    for c in (0, 17, 127):
        q = np.zeros(D); q[c] = 3.0
        k = np.zeros(D); k[c] = -5.0
        before = np.sum(q ** 2 * k ** 2)
        after = np.sum((q @ R) ** 2 * (k @ R) ** 2)
        assert before / after == pytest.approx(g["value"], rel=1e-12)


def test_descale_closed_form():
    """Smallest power of two d with amax <= 448 d."""
    assert OQ.descale_for(0.0) == 1.0
    assert OQ.descale_for(448.0) == 1.0
    assert OQ.descale_for(448.0 * (1 + 2 ** -40)) == 2.0
    assert OQ.descale_for(224.0) == 0.5
    assert OQ.descale_for(224.0 * (1 + 2 ** -40)) == 1.0
    assert OQ.descale_for(2.0 ** -140) == 2.0 ** -126        # FP32-normal floor
    assert OQ.descale_for(448.0 * 2.0 ** -126) == 2.0 ** -126
    rng = np.random.default_rng(0)
    for a in 10.0 ** rng.uniform(-30, 30, 2000):
        d = OQ.descale_for(a)
        assert OQ.is_pow2(d)
        assert 224.0 < a / d <= 448.0


def _midpoint_distance(z):
    """|z - nearest e4m3 rounding midpoint| / |z| (midpoints of codes 0..126)."""
    vals = bf.e4m3_values()[:127]
    mids = 0.5 * (vals[:-1] + vals[1:])
    a = np.abs(z)
    i = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    d = np.minimum(np.abs(a - mids[i - 1]), np.abs(a - mids[i]))
    return d / np.maximum(a, 1e-300)


@pytest.mark.parametrize("rot", [False, True])
@pytest.mark.parametrize("smooth", [False, True])
def test_codes_match_torch_cast(rot, smooth):
    """Every code equals PyTorch's float8_e4m3fn cast of float32(z), where
    float32 rounding of z cannot move it across a midpoint."""
    x = _bf16((2, 64, 3, 128), 11, 2.5)
    s = S.rotation_signs(128) if rot else None
    r = OQ.quantize(x, s, smooth)
    z = r["z"]
    tor = torch.from_numpy(z.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    if rot or smooth:
        safe = _midpoint_distance(z) > 2.0 ** -22
        assert np.mean(safe) > 0.999
    else:
        # BF16 / 2^k is exact in float32, and many values sit exactly on a
        # midpoint: every code, ties included, must match
        safe = np.ones(z.shape, dtype=bool)
        assert np.mean(_midpoint_distance(z) == 0) > 0.01
    assert np.array_equal(r["codes"][safe], tor[safe])
    assert OQ.is_pow2(r["descale"])
    assert 224.0 < np.max(np.abs(z)) <= 448.0


def test_dynamic_scale_uses_transformed_amax():
    """Sec. V-A: FP8 scales are computed after the rotation."""
    x = _bf16((1, 128, 2, 128), 12)
    s = S.rotation_signs(128)
    r = OQ.quantize(x, s)
    y = OQ.bf16_bits_to_f64(x).reshape(-1, 128) @ OQ.rotation(s)
    assert r["amax"] == pytest.approx(np.max(np.abs(y)), rel=0, abs=0)
    assert r["descale"] == OQ.descale_for(np.max(np.abs(y)))


def test_static_scale_saturates_and_special_values():
    x = S.to_bf16_bits(np.array([0.0, 1.0, -3.0, 500.0, -1e5, np.inf, -np.inf, np.nan],
                                dtype=np.float32)).reshape(1, 1, 1, 8)
    r = OQ.quantize(x, None, False, static_descale=1.0)
    assert list(r["codes"].reshape(-1)) == [0x00, 0x38, 0xC4, 0x7E, 0xFE, 0x7E, 0xFE, 0x7F]
    with pytest.raises(ValueError):
        OQ.quantize(x, None, False, static_descale=3.0)
    # a dynamic scale ignores the non-finite elements
    r = OQ.quantize(x, None, False)
    big = float(OQ.bf16_bits_to_f64(x).reshape(-1)[4])      # BF16 of -1e5
    assert r["amax"] == -big and r["descale"] == 256.0


def _attn(q, k, v):
    """Causal fp64 attention on float64 [B, N, H, D] arrays, c = 1/sqrt(d)."""
    B, N, Hq, D = q.shape
    grp = Hq // k.shape[2]
    out = np.zeros((B, N, Hq, v.shape[3]))
    mask = np.tril(np.ones((N, N), dtype=bool))
    for b in range(B):
        for h in range(Hq):
            s = (q[b, :, h] @ k[b, :, h // grp].T) / math.sqrt(D)
            s = np.where(mask, s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            out[b, :, h] = (p / p.sum(axis=1, keepdims=True)) @ v[b, :, h // grp]
    return out


@pytest.mark.parametrize("D", [128, 192])
def test_rotation_and_smoothing_leave_attention_unchanged(D):
    """Sec. V-A: rotation keeps QK^T; subtracting the mean key lowers every
    score of a query row by the same value, which the softmax cancels
    (footnote 18).  So fp64 attention on the unrounded transformed Q, K
    equals fp64 attention on Q, K."""
    wl = S.Workload("t", 1, 4, 2, 96, D, 128, kind="kbias")
    q, k, v, _ = S.fp32_qkv(wl, seed=5)
    qb, kb = S.to_bf16_bits(q), S.to_bf16_bits(k)
    s = S.rotation_signs(D)
    rq = OQ.quantize(qb, s, False)
    rk = OQ.quantize(kb, s, True)
    qt = rq["z"] * rq["descale"]
    kt = rk["z"] * rk["descale"]
    vv = v.astype(np.float64)
    ref = _attn(OQ.bf16_bits_to_f64(qb), OQ.bf16_bits_to_f64(kb), vv)
    got = _attn(qt, kt, vv)
    assert np.max(np.abs(got - ref)) < 1e-11
    # the smoothed, rotated keys have zero mean over the sequence
    assert np.max(np.abs(kt.mean(axis=1))) < 1e-12 * np.max(np.abs(kt))
    assert np.allclose(rk["mean"], OQ.bf16_bits_to_f64(kb).mean(axis=1), rtol=0, atol=1e-15)


def _input_error(wl, seed, rot, smooth):
    """Relative RMS error of fp64 attention on the e4m3 inputs against fp64
    attention on the BF16 inputs (the "input" term of Table XIII)."""
    q, k, v, _ = S.fp32_qkv(wl, seed=seed)
    qb, kb, vb = S.to_bf16_bits(q), S.to_bf16_bits(k), S.to_bf16_bits(v)
    s = S.rotation_signs(wl.d_qk) if rot else None
    rq = OQ.quantize(qb, s, False)
    rk = OQ.quantize(kb, s, smooth)
    rv = OQ.quantize(vb, None, False)
    dec = bf.e4m3_values()
    got = _attn(dec[rq["codes"]] * rq["descale"], dec[rk["codes"]] * rk["descale"],
                dec[rv["codes"]] * rv["descale"])
    ref = _attn(OQ.bf16_bits_to_f64(qb), OQ.bf16_bits_to_f64(kb), OQ.bf16_bits_to_f64(vb))
    return np.sqrt(np.mean((got - ref) ** 2) / np.mean(ref ** 2))


def test_table13_rotation_lowers_input_error_on_outlier_channels(golden):
    """Table XIII: rotating Q and K roughly halves the input error on heads
    whose q and k share large channels.  The activation-like inputs have 4
    such channels per KV head (x20)."""
    wl = S.Workload("act", 1, 4, 1, 256, 128, 128, kind="activation")
    e0 = _input_error(wl, 21, False, False)
    e1 = _input_error(wl, 21, True, False)
    lo, hi = golden["table13_rotation_input_error_ratio"]["range"]
    print("input error none / rotation:", e0, e1, e1 / e0)
    assert e1 / e0 < hi


def test_k_smoothing_lowers_input_error_on_offset_keys():
    """Table XIII: K smoothing lowers the error further when the keys share
    a large mean (here an N(0, 16) offset per KV head and channel)."""
    wl = S.Workload("kb", 1, 4, 2, 256, 128, 128, kind="kbias")
    e1 = _input_error(wl, 22, True, False)
    e2 = _input_error(wl, 22, True, True)
    print("input error rotation / rotation+smoothing:", e1, e2)
    assert e2 < 0.8 * e1
