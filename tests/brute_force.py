"""Independent brute-force restatement of the method, for tiny inputs only.

Used to pin the C oracle.  It shares no code with it and computes each step
another way:

* e4m3 rounding by enumerating every finite code and taking the nearest
  value (ties to the even code), instead of exponent/mantissa arithmetic;
* BF16 rounding with exact rational arithmetic (``fractions.Fraction``);
* the whole score matrix as one float64 matmul;
* for the running maximum, the reference maximum of every key block is
  computed first and the blocks are combined at the end with factors
  2^(m_block - m_last), instead of rescaling an accumulator as it goes.

Source: "ZYFA: Speed and Accuracy of FP8 FlashAttention on AMD CDNA4",
Sec. II-B, II-C, IV-A (lazy rescaling), IV-B1 (Eq. 2), IV-B2, IV-B3, V-D.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


def e4m3_values() -> np.ndarray:
    """Value of every code 0..255 from its bit fields (NaN for 0x7F, 0xFF)."""
    vals = np.empty(256)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            vals[c] = np.nan
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        vals[c] = -mag if s else mag
    return vals


_VALS = e4m3_values()
_POS = _VALS[:127]          # codes 0..126, increasing


def e4m3_encode(x: float) -> int:
    """Nearest finite e4m3 code by enumeration, ties to the even code,
    saturating beyond 448; NaN -> 0x7F."""
    if math.isnan(x):
        return 0x7F
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    d = np.abs(_POS - a)
    best = np.flatnonzero(d == d.min())
    code = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
    return sign | code


def bf16_round(x: float) -> float:
    """Round a float to BF16 (8 significant bits) with exact rationals."""
    if x == 0.0 or math.isnan(x) or math.isinf(x):
        return x
    sign = -1.0 if x < 0 else 1.0
    a = Fraction(abs(x))
    e = math.floor(math.log2(abs(x)))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** max(e - 7, -133)
    n = a / ulp
    lo = math.floor(n)
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * float(lo * ulp)


def lean_code(u: float, sigma: float, beta: float) -> int:
    y = 8.0 * (u + sigma + 7.0) - beta
    if not y > 0:
        return 0
    return int(min(np.rint(y), 255))


def prob(u, dtype, p_mode, sigma, beta):
    """(rounded, unrounded) probability for u = x + o."""
    exact = 2.0 ** (u + sigma)
    if p_mode == 2:
        return exact, exact
    if dtype == "bf16":
        return bf16_round(exact), exact
    if p_mode == 1:
        return _VALS[lean_code(u, sigma, beta)], exact
    return _VALS[e4m3_encode(exact)], exact


def decode(a, dtype):
    if dtype == "e4m3":
        return _VALS[np.asarray(a, dtype=np.uint8)]
    b = np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def forward(q, k, v, *, dtype, descale, p_mode, block_scale, max_mode, tau,
            kv_block, scale_block, denom_mode, sigma, beta, softmax_scale,
            o_max=127, key_begin=0, key_end=None):
    """Full (B, N, Hq, d_v) output in float64, all rows, causal.  dtype
    'mixed': BF16 Q and K, e4m3 V and e4m3 probabilities."""
    B, N, Hq, dqk = q.shape
    Hkv, dv_ = k.shape[2], v.shape[3]
    grp = Hq // Hkv
    qk_dtype = "bf16" if dtype == "mixed" else dtype
    v_dtype = "e4m3" if dtype == "mixed" else dtype
    Q, K, V = decode(q, qk_dtype), decode(k, qk_dtype), decode(v, v_dtype)
    dtype = v_dtype
    dq, dk, dvs = descale
    out = np.zeros((B, N, Hq, dv_))
    for b in range(B):
        for h in range(Hq):
            g = h // grp
            T = (Q[b, :, h, :] @ K[b, :, g, :].T) * (softmax_scale * dq * dk / math.log(2.0))
            for i in range(N):
                kb = key_begin
                ke = i + 1 if key_end is None else min(i + 1, key_end)
                if ke <= kb:
                    continue                       # nothing visible: output 0
                t = T[i, kb:ke]
                nk = ke - kb
                if max_mode == 0:
                    segs = [(0, nk, float(np.max(t)))]
                else:
                    segs, m = [], None
                    for s0 in range(0, nk, kv_block):
                        s1 = min(s0 + kv_block, nk)
                        bm = float(np.max(t[s0:s1]))
                        if m is None or bm - m > tau:
                            m = bm
                        segs.append((s0, s1, m))
                m_last = segs[-1][2]
                num = np.zeros(dv_)
                den = 0.0
                for s0, s1, m in segs:
                    f = 2.0 ** (m - m_last)
                    for j in range(s0, s1):
                        c0 = (j // scale_block) * scale_block
                        lo, hi = max(c0, s0), min(c0 + scale_block, s1)
                        hm = float(np.max(t[lo:hi]))
                        o = int(min(max(math.floor(m - hm), 0), o_max)) if block_scale else 0
                        pr, pu = prob(t[j] - m + o, dtype, p_mode, sigma, beta)
                        w = pr * 2.0 ** -o
                        num += f * w * V[b, kb + j, g, :]
                        den += f * (w if denom_mode == 0 else pu * 2.0 ** -o)
                out[b, i, h, :] = dvs * num / den
    return out


def attention_fp64(q, k, v, *, dtype, descale, softmax_scale):
    """softmax(c Q K^T + causal mask) V in float64 on the dequantised inputs."""
    B, N, Hq, _ = q.shape
    Hkv = k.shape[2]
    grp = Hq // Hkv
    qk_dtype = "bf16" if dtype == "mixed" else dtype
    v_dtype = "e4m3" if dtype == "mixed" else dtype
    Q, K, V = decode(q, qk_dtype), decode(k, qk_dtype), decode(v, v_dtype)
    dq, dk, dvs = descale
    out = np.zeros((B, N, Hq, v.shape[3]))
    mask = np.tril(np.ones((N, N), dtype=bool))
    for b in range(B):
        for h in range(Hq):
            g = h // grp
            S = (Q[b, :, h, :] @ K[b, :, g, :].T) * (softmax_scale * dq * dk)
            S = np.where(mask, S, -np.inf)
            S = S - S.max(axis=1, keepdims=True)
            P = np.exp(S)
            P /= P.sum(axis=1, keepdims=True)
            out[b, :, h, :] = dvs * (P @ V[b, :, g, :])
    return out
