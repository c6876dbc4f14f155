"""CPU oracle of the quantisation pass that feeds FP8 attention.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  The
product path never imports it, and the two share no code.

What it computes ("ZYFA: Speed and Accuracy of FP8 FlashAttention on AMD
CDNA4", Sec. V-A, paragraphs "FP8 inputs and policies" and "Rotation and K
smoothing", with footnotes 17, 18 and 25, and Table XIII):

1. K smoothing (optional): subtract from every key the mean key of its head
   over the sequence.  Read here as the mean over the N positions of one
   (batch, head) pair, each channel separately.
2. Rotation (optional): multiply each row vector by one orthogonal matrix
   R = diag(s) (C_m kron H_{D/m}), with s a vector of random signs, H the
   normalised Sylvester-Hadamard matrix and C_m the orthonormal DCT-II of
   size m; m = 1 for D = 128 and m = 3 for D = 192 (read as: m is the odd
   part of D).  The pages draw s "with seed 0" from an unnamed generator, so
   s is an input here.  The Kronecker product takes C's index as the major
   one: R[a*(D/m) + b, a'*(D/m) + b'] = s[a*(D/m) + b] C[a, a'] H[b, b'],
   with C[k, n] = sqrt((2 - [k = 0]) / m) cos(pi (2n + 1) k / (2m)).
3. Per-tensor power-of-two descale, computed after the transforms: per call
   ("dynamic"), the smallest power of two d with amax <= 448 d, where amax is
   the largest finite |value| of the transformed tensor (d = 1 when amax is
   0; d is kept at or above 2^-126 so that d and 1/d are normal FP32
   numbers); or static, a power of two given by the caller.
4. Codes: e4m3 round-to-nearest-even of value / d, saturating to +-448 (so a
   static scale that the tensor outgrows clips it); NaN -> 0x7F.

The kernel does these steps in FP32 (the pages multiply in FP32); this
oracle does them in float64, so it gives the exact value that each FP32
result approximates.  The parity tests accept a kernel code that differs
from the oracle's only where the exact value lies within a stated FP32 error
bound of the rounding midpoint between the two codes.

Pins: tests/test_oracle_quantize.py (SciPy's Hadamard matrix and DCT, a
butterfly Walsh-Hadamard transform, orthogonality, softmax invariance of
rotation and smoothing, footnote 25's factor of 128, the closed form of the
descale, PyTorch's e4m3 cast, and the direction of Table XIII).
"""
from __future__ import annotations

import math

import numpy as np

from . import e4m3_encode_array

E4M3_MAX = 448.0


def odd_part(D: int) -> int:
    """m of the rotation: D = m * 2^k with m odd (1 for 128, 3 for 192)."""
    m = int(D)
    if m <= 0:
        raise ValueError("D must be positive")
    while m % 2 == 0:
        m //= 2
    return m


def hadamard(n: int) -> np.ndarray:
    """Normalised Sylvester-Hadamard matrix H_n (n a power of two):
    H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]] / sqrt(2)."""
    if n < 1 or n & (n - 1):
        raise ValueError("Sylvester's construction needs a power of two")
    H = np.ones((1, 1))
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]]) / math.sqrt(2.0)
    return H


def dct2(m: int) -> np.ndarray:
    """Orthonormal DCT-II matrix C_m, C[k, n] = w_k cos(pi (2n+1) k / (2m)),
    w_0 = sqrt(1/m), w_k = sqrt(2/m) otherwise."""
    k = np.arange(m)[:, None]
    n = np.arange(m)[None, :]
    C = np.cos(math.pi * (2 * n + 1) * k / (2.0 * m))
    w = np.full((m, 1), math.sqrt(2.0 / m))
    w[0, 0] = math.sqrt(1.0 / m)
    return w * C


def rotation(signs) -> np.ndarray:
    """R = diag(s) (C_m kron H_{D/m}) for the sign vector s (length D)."""
    s = np.asarray(signs, dtype=np.float64).reshape(-1)
    if not np.all(np.abs(s) == 1.0):
        raise ValueError("signs must be +1 or -1")
    D = s.size
    m = odd_part(D)
    return s[:, None] * np.kron(dct2(m), hadamard(D // m))


MIN_DESCALE_EXP = -126


def descale_for(amax: float) -> float:
    """Smallest power of two d >= 2^-126 with amax <= 448 d (1 when amax is
    0).  The floor keeps d and 1/d normal FP32 numbers (the descale is an
    FP32 value, Sec. II-C); it matters only for amax below about 2^-117."""
    if not amax > 0.0:
        return 1.0
    e = math.frexp(amax)[1] - 1            # amax in [2^e, 2^(e+1))
    e -= 8                                 # 448 = 1.75 * 2^8
    while amax > E4M3_MAX * 2.0 ** e:
        e += 1
    while e > MIN_DESCALE_EXP and amax <= E4M3_MAX * 2.0 ** (e - 1):
        e -= 1
    return 2.0 ** max(e, MIN_DESCALE_EXP)


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def is_pow2(x: float) -> bool:
    return x > 0.0 and math.isfinite(x) and math.frexp(x)[0] == 0.5


def quantize(x_bits, signs=None, smooth: bool = False, static_descale=None,
             rows=None, chunk: int = 1 << 16):
    """Quantise a BF16 tensor [B, N, H, D] (given as uint16 bits).

    Returns a dict with
      ``descale``  the per-tensor descale d;
      ``amax``     largest finite |transformed value| (None for static d);
      ``mean``     [B, H, D] float64 means subtracted (None without smoothing);
      ``z``        float64 transformed value / d for the selected rows;
      ``codes``    uint8 e4m3 codes of ``z``;
      ``rows``     flat row ids ((b*N + n)*H + h) that ``z``/``codes`` hold
                   (all rows when ``rows`` is None, then shaped like x).
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    if x_bits.ndim != 4:
        raise ValueError("x must be [B, N, H, D]")
    B, N, H, D = x_bits.shape
    flat = x_bits.reshape(B * N * H, D)
    R = rotation(signs) if signs is not None else None

    mean = None
    if smooth:
        x = bf16_bits_to_f64(x_bits)
        mean = x.mean(axis=1) if N > 0 else np.zeros((B, H, D))      # [B, H, D]
        del x
    mean_rows = None if mean is None else mean.reshape(B * H, D)

    def transform(ids):
        y = bf16_bits_to_f64(flat[ids])
        if mean_rows is not None:
            b = ids // (N * H)
            h = ids % H
            y = y - mean_rows[b * H + h]
        if R is not None:
            y = y @ R
        return y

    if static_descale is not None:
        d = float(static_descale)
        if not (is_pow2(d) and 2.0 ** MIN_DESCALE_EXP <= d <= 2.0 ** 127):
            raise ValueError("a static descale must be a power of two in [2^-126, 2^127]")
        amax = None
    else:
        amax = 0.0
        total = B * N * H
        for s0 in range(0, total, chunk):
            y = np.abs(transform(np.arange(s0, min(total, s0 + chunk))))
            fin = y[np.isfinite(y)]
            if fin.size:
                amax = max(amax, float(fin.max()))
        d = descale_for(amax)

    all_rows = rows is None
    ids = np.arange(B * N * H) if all_rows else np.asarray(rows, dtype=np.int64)
    z = np.empty((ids.size, D))
    for s0 in range(0, ids.size, chunk):
        z[s0:s0 + chunk] = transform(ids[s0:s0 + chunk]) / d
    codes = e4m3_encode_array(z)
    if all_rows:
        z = z.reshape(B, N, H, D)
        codes = codes.reshape(B, N, H, D)
    return {"descale": d, "amax": amax, "mean": mean, "z": z, "codes": codes,
            "rows": ids}
