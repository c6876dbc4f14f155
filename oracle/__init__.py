"""CPU oracle for causal FP8 / BF16 flash attention (ZYFA method).

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  The
product path (``fp8_causal_flashattention_gb300``) never imports it, and the
two share no code.

The arithmetic lives in ``zyfa_oracle.c`` (plain C, fp64, -ffp-contract=off);
this module compiles it with gcc on first use and marshals numpy arrays.

Which passage each parameter follows ("ZYFA: Speed and Accuracy of FP8
FlashAttention on AMD CDNA4"):

* ``sigma`` = 6 and ``beta`` = 0.35: Sec. IV-B1, Eq. (2) (Lean P);
* ``block_scale`` and ``scale_block`` = 64: Sec. IV-B2, Fig. 5;
* ``denom_mode`` 0 (sum of the rounded probabilities): Sec. IV-B3, fn. 12;
* ``max_mode`` 1 with ``tau`` (0.125 FP8; 0.5 BF16 d=128; 8 BF16 d=192) and
  ``kv_block`` = 128: the running maximum with lazy rescaling, Sec. II-B and
  Sec. IV-A "Lazy rescaling";
* ``max_mode`` 0: the exact row maximum used to emulate the P term,
  Sec. V-E "Error of each stage of one call";
* ``attn_fp64``: fp64 attention on the quantised inputs, Sec. V-D, fn. 15;
* ``key_begin`` / ``key_end`` and ``merge``: partial attention over a key
  range and the merge of partial results by their LSE (Sec. IV-B3: the LSE
  lets results over different key ranges be merged); the running maximum of
  a range starts at its first key;
* ``dtype='mixed'``: BF16 QK^T with the FP8 PV path, the variant the
  conclusion recommends (keep QK^T in BF16, run only PV in FP8); read as the
  e4m3 method (tau = 0.125, sigma = 6, block scaling, rounded denominator)
  with scores from BF16 Q and K and no Q/K descale;
* ``quantize`` (oracle/quantize.py): the quantisation pass before the
  kernel -- K smoothing, the rotation R = diag(s)(C_m kron H_{D/m}) and the
  per-tensor power-of-two descale, Sec. V-A "FP8 inputs and policies" and
  "Rotation and K smoothing", Table XIII.

Parity pins: see tests/test_oracle_*.py (brute force, printed constants,
closed forms and invariants).  No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zyfa_oracle.c")
_LIB = os.path.join(_HERE, "libzyfa_oracle.so")
_lock = threading.Lock()
_lib = None

P_EXACT, P_LEAN, P_UNROUNDED = 0, 1, 2
MAX_EXACT, MAX_RUNNING = 0, 1
DENOM_ROUNDED, DENOM_UNROUNDED = 0, 1

SIGMA_FP8 = 6.0
BETA = 0.35
TAU_FP8 = 0.125
KV_BLOCK = 128
SCALE_BLOCK = 64
O_MAX = 127


def tau_bf16(d_qk: int) -> float:
    """Lazy-rescaling threshold of the BF16 kernels (Sec. IV-A)."""
    return 8.0 if d_qk == 192 else 0.5


class Params(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int),
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("N", ctypes.c_int), ("d_qk", ctypes.c_int), ("d_v", ctypes.c_int),
        ("causal", ctypes.c_int),
        ("descale_q", ctypes.c_double), ("descale_k", ctypes.c_double),
        ("descale_v", ctypes.c_double),
        ("softmax_scale", ctypes.c_double),
        ("p_mode", ctypes.c_int), ("block_scale", ctypes.c_int),
        ("max_mode", ctypes.c_int), ("tau", ctypes.c_double),
        ("kv_block", ctypes.c_int), ("scale_block", ctypes.c_int),
        ("denom_mode", ctypes.c_int),
        ("sigma", ctypes.c_double), ("beta", ctypes.c_double),
        ("o_max", ctypes.c_int),
        ("key_begin", ctypes.c_int), ("key_end", ctypes.c_int),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (no GPU needed)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared",
               "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC,
               "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.zo_e4m3_decode.restype = ctypes.c_double
        lib.zo_e4m3_decode.argtypes = [ctypes.c_uint]
        lib.zo_e4m3_encode.restype = ctypes.c_uint
        lib.zo_e4m3_encode.argtypes = [ctypes.c_double]
        lib.zo_e4m3_encode_n.restype = None
        lib.zo_e4m3_encode_n.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_longlong]
        lib.zo_bf16_encode.restype = ctypes.c_uint
        lib.zo_bf16_encode.argtypes = [ctypes.c_double]
        lib.zo_bf16_decode.restype = ctypes.c_double
        lib.zo_bf16_decode.argtypes = [ctypes.c_uint]
        lib.zo_lean_y.restype = ctypes.c_double
        lib.zo_lean_y.argtypes = [ctypes.c_double] * 3
        lib.zo_lean_code.restype = ctypes.c_uint
        lib.zo_lean_code.argtypes = [ctypes.c_double] * 3
        lib.zo_exact_code.restype = ctypes.c_uint
        lib.zo_exact_code.argtypes = [ctypes.c_double] * 2
        vp = ctypes.c_void_p
        lib.zo_fwd.restype = ctypes.c_int
        lib.zo_fwd.argtypes = [ctypes.POINTER(Params), vp, vp, vp, vp,
                               ctypes.c_longlong, vp, vp, vp, ctypes.c_int]
        lib.zo_attn_fp64.restype = ctypes.c_int
        lib.zo_attn_fp64.argtypes = [ctypes.POINTER(Params), vp, vp, vp, vp,
                                     ctypes.c_longlong, vp, vp, ctypes.c_int]
        _lib = lib
    return _lib


# --------------------------------------------------------------------------
# scalar codecs (exposed for the pins)
# --------------------------------------------------------------------------
def e4m3_decode(code: int) -> float:
    return _load().zo_e4m3_decode(int(code))


def e4m3_encode(x: float) -> int:
    return int(_load().zo_e4m3_encode(float(x)))


def e4m3_encode_array(x) -> np.ndarray:
    """zo_e4m3_encode applied to every element of a float64 array."""
    xa = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(xa.shape, dtype=np.uint8)
    _load().zo_e4m3_encode_n(xa.ctypes.data, out.ctypes.data, xa.size)
    return out


def bf16_encode(x: float) -> int:
    return int(_load().zo_bf16_encode(float(x)))


def bf16_decode(bits: int) -> float:
    return _load().zo_bf16_decode(int(bits))


def lean_y(u: float, sigma: float = SIGMA_FP8, beta: float = BETA) -> float:
    return _load().zo_lean_y(float(u), float(sigma), float(beta))


def lean_code(u: float, sigma: float = SIGMA_FP8, beta: float = BETA) -> int:
    return int(_load().zo_lean_code(float(u), float(sigma), float(beta)))


def exact_code(u: float, sigma: float = SIGMA_FP8) -> int:
    return int(_load().zo_exact_code(float(u), float(sigma)))


def e4m3_decode_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


# --------------------------------------------------------------------------
# forward
# --------------------------------------------------------------------------
def make_params(*, dtype: str, B: int, Hq: int, Hkv: int, N: int, d_qk: int,
                d_v: int, descale=(1.0, 1.0, 1.0), softmax_scale=None,
                p_mode: int = P_LEAN, block_scale: int = 1,
                max_mode: int = MAX_RUNNING, tau=None, kv_block: int = KV_BLOCK,
                scale_block: int = SCALE_BLOCK, denom_mode=None, sigma=None,
                beta: float = BETA, causal: int = 1, o_max: int = O_MAX,
                key_begin: int = 0, key_end: int = -1) -> Params:
    """Parameters with the method's defaults for ``dtype``: 'e4m3', 'bf16', or
    'mixed' (BF16 Q and K, e4m3 V: the FP8 probability path of the e4m3
    kernels after a BF16 QK^T; Q and K carry no descale)."""
    mixed = dtype == "mixed"
    fp8 = dtype == "e4m3" or mixed
    if not fp8 and dtype != "bf16":
        raise ValueError(dtype)
    if softmax_scale is None:
        softmax_scale = 1.0 / np.sqrt(d_qk)
    if tau is None:
        tau = TAU_FP8 if fp8 else tau_bf16(d_qk)
    if denom_mode is None:
        denom_mode = DENOM_ROUNDED if fp8 else DENOM_UNROUNDED
    if sigma is None:
        sigma = SIGMA_FP8 if fp8 else 0.0
    if not fp8:
        descale = (1.0, 1.0, 1.0)
        block_scale = 0
    if mixed:
        descale = (1.0, 1.0, descale[2])
    return Params(2 if mixed else (0 if fp8 else 1), B, Hq, Hkv, N, d_qk, d_v, int(causal),
                  float(descale[0]), float(descale[1]), float(descale[2]),
                  float(softmax_scale), int(p_mode), int(block_scale),
                  int(max_mode), float(tau), int(kv_block), int(scale_block),
                  int(denom_mode), float(sigma), float(beta), int(o_max),
                  int(key_begin), int(key_end))


def _prep(p: Params, q, k, v, rows):
    qk_t = np.uint8 if p.dtype == 0 else np.uint16
    v_t = np.uint16 if p.dtype == 1 else np.uint8
    arrs = []
    for a, h, d, want in ((q, p.Hq, p.d_qk, qk_t), (k, p.Hkv, p.d_qk, qk_t), (v, p.Hkv, p.d_v, v_t)):
        a = np.ascontiguousarray(a)
        if a.dtype != want:
            a = a.view(want)
        if a.size != p.B * p.N * h * d:
            raise ValueError("tensor size does not match B*N*H*d")
        arrs.append(a)
    if rows is None:
        rows = np.arange(p.B * p.Hq * p.N, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    return arrs, rows


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def fwd(p: Params, q, k, v, rows=None, nthreads=None):
    """Run the method on ``rows`` (flat (b*Hq + h)*N + i; all rows if None).

    Returns ``(out_f64, out_bf16_bits, lse)`` with shapes (R, d_v), (R, d_v),
    (R,).  Inputs are e4m3 codes (uint8) or BF16 bits (uint16) in BSHD order.
    """
    lib = _load()
    (qa, ka, va), rows = _prep(p, q, k, v, rows)
    R = rows.size
    out = np.empty((R, p.d_v), dtype=np.float64)
    outb = np.empty((R, p.d_v), dtype=np.uint16)
    lse = np.empty((R,), dtype=np.float64)
    rc = lib.zo_fwd(ctypes.byref(p), qa.ctypes.data, ka.ctypes.data,
                    va.ctypes.data, rows.ctypes.data, R, out.ctypes.data,
                    outb.ctypes.data, lse.ctypes.data,
                    nthreads or default_threads())
    if rc:
        raise ValueError(f"oracle zo_fwd failed with status {rc}")
    return out, outb, lse


def attn_fp64(p: Params, q, k, v, rows=None, nthreads=None):
    """fp64 softmax attention on the dequantised inputs: ``(out, lse)``."""
    lib = _load()
    (qa, ka, va), rows = _prep(p, q, k, v, rows)
    R = rows.size
    out = np.empty((R, p.d_v), dtype=np.float64)
    lse = np.empty((R,), dtype=np.float64)
    rc = lib.zo_attn_fp64(ctypes.byref(p), qa.ctypes.data, ka.ctypes.data,
                          va.ctypes.data, rows.ctypes.data, R, out.ctypes.data,
                          lse.ctypes.data, nthreads or default_threads())
    if rc:
        raise ValueError(f"oracle zo_attn_fp64 failed with status {rc}")
    return out, lse


def merge(outs, lses):
    """Combine partial attention results over disjoint key ranges (Sec. IV-B3:
    the LSE is returned so that results over different key ranges can be
    merged): with L = ln sum_i exp(LSE_i), O = sum_i exp(LSE_i - L) O_i.  Rows
    that no range reaches get O = 0 and L = -inf.  float64 throughout."""
    outs = [np.asarray(o, dtype=np.float64) for o in outs]
    lses = np.stack([np.asarray(l, dtype=np.float64) for l in lses])     # [P, R]
    top = np.max(lses, axis=0)
    live = np.isfinite(top)
    safe = np.where(live, top, 0.0)
    w = np.exp(lses - safe)                                             # exp(-inf) = 0
    tot = w.sum(axis=0)
    L = np.where(live, safe + np.log(np.where(live, tot, 1.0)), -np.inf)
    out = np.zeros_like(outs[0])
    for wi, oi in zip(w, outs):
        out += np.where(live, wi / np.where(live, tot, 1.0), 0.0)[:, None] * oi
    return out, L


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
