"""Seeded synthetic inputs shared by the tests, the bench and the oracle legs.

This module holds none of the attention method's arithmetic: it draws
Gaussian tensors from a counter-based generator, casts them to e4m3 or BF16
with PyTorch's own conversions, and lists the workload shapes.

Generator: SplitMix64 (S. Vigna's published finaliser, constants
0x9E3779B97F4A7C15, 0xBF58476D1CE4E5B9, 0x94D049BB133111EB) used as a
counter-based stream -- element n of stream (seed, id) depends only on
(seed, id, n) -- followed by the Box-Muller transform.  Element 2n takes the
cosine branch and 2n+1 the sine branch of counter pair (2n, 2n+1).

Quantisation recipe (the workloads' own input recipe): per-tensor descale =
amax / 448, code = e4m3(x / descale) rounded by ``torch.Tensor.to(
torch.float8_e4m3fn)`` (round to nearest even).  BF16 inputs are
``x.to(torch.bfloat16)``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
from dataclasses import dataclass, field

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)
E4M3_MAX = 448.0
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * M1
    z = (z ^ (z >> np.uint64(27))) * M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        z = np.array([(int(seed) << 16) + int(stream)], dtype=np.uint64)
        return _mix(z + GAMMA)[0]


def _normal_chunk(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Normals for elements [start, start+count); start and count even."""
    pairs = count // 2
    n0 = start // 2
    with np.errstate(over="ignore"):
        c = np.arange(2 * n0, 2 * (n0 + pairs), dtype=np.uint64)
        u = _mix(key + (c + np.uint64(1)) * GAMMA)
    u = ((u >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    ang = 2.0 * np.pi * u2
    out = np.empty(count, dtype=np.float32)
    out[0::2] = r * np.cos(ang)
    out[1::2] = r * np.sin(ang)
    return out


def normal(shape, seed: int, stream: int, threads: int | None = None) -> np.ndarray:
    """float32 N(0,1) tensor of ``shape``; element n (flat, C order) depends
    only on (seed, stream, n)."""
    total = int(np.prod(shape))
    out = np.empty(total + (total & 1), dtype=np.float32)
    key = _key(seed, stream)
    starts = list(range(0, out.size, _CHUNK))

    def job(s):
        cnt = min(_CHUNK, out.size - s)
        out[s:s + cnt] = _normal_chunk(key, s, cnt)

    if len(starts) == 1:
        job(0)
    else:
        with cf.ThreadPoolExecutor(threads or min(32, os.cpu_count() or 1)) as ex:
            list(ex.map(job, starts))
    return out[:total].reshape(shape)


STREAM_SIGNS = 100


def rotation_signs(D: int, seed: int = 0) -> np.ndarray:
    """float32 vector of D random signs (+1/-1): sign j is the top bit of
    SplitMix64 counter j of stream (seed, STREAM_SIGNS)."""
    key = _key(seed, STREAM_SIGNS)
    with np.errstate(over="ignore"):
        c = np.arange(D, dtype=np.uint64)
        u = _mix(key + (c + np.uint64(1)) * GAMMA)
    return np.where((u >> np.uint64(63)) == 0, 1.0, -1.0).astype(np.float32)


def quantize_e4m3(x: np.ndarray):
    """Per-tensor e4m3 quantisation: returns (codes uint8, descale float)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    amax = float(t.abs().max()) if t.numel() else 1.0
    descale = np.float32(amax / E4M3_MAX) if amax > 0 else np.float32(1.0)
    codes = (t / torch.tensor(float(descale), dtype=torch.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8)
    return codes.numpy(), float(descale)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d_qk: int
    d_v: int
    kind: str = "gaussian"          # "gaussian", "activation", "sink", "kbias" or FIG15_KINDS
    note: str = ""

    @property
    def causal_flops(self) -> float:
        """F = 2*B*Hq*N^2*(d_qk+d_v)/2 (Eq. 1 of the paper)."""
        return float(self.B) * self.Hq * self.N * self.N * (self.d_qk + self.d_v)

    def shapes(self):
        return ((self.B, self.N, self.Hq, self.d_qk),
                (self.B, self.N, self.Hkv, self.d_qk),
                (self.B, self.N, self.Hkv, self.d_v))


WORKLOADS = {
    "pr1": Workload("pr1", 1, 1, 1, 256, 128, 128,
                    note="B=1 H=1 N=256 d=128, all rows checked"),
    "d128": Workload("d128", 1, 32, 32, 32768, 128, 128,
                     note="kernel bench d=128, N=32K, 32 heads"),
    "mla": Workload("mla", 1, 128, 128, 32768, 192, 128,
                    note="MLA prefill shape d_qk=192 d_v=128, N=32K, 128 heads"),
    "gqa_act": Workload("gqa_act", 2, 32, 8, 8192, 128, 128, kind="activation",
                        note="activation-like GQA, outlier channels"),
    "sweep_1k": Workload("sweep_1k", 64, 16, 16, 1024, 128, 128),
    "sweep_4k": Workload("sweep_4k", 16, 16, 16, 4096, 128, 128),
    "sweep_16k": Workload("sweep_16k", 4, 16, 16, 16384, 128, 128),
    "sweep_64k": Workload("sweep_64k", 1, 16, 16, 65536, 128, 128),
}

SEED = 0
STREAM_Q, STREAM_K, STREAM_V = 0, 1, 2
ROW_SAMPLE_SEED = 1234


@dataclass
class Inputs:
    """One synthetic problem: e4m3 codes + descales and/or BF16 bits."""
    wl: Workload
    q8: np.ndarray | None = None
    k8: np.ndarray | None = None
    v8: np.ndarray | None = None
    descale: tuple = (1.0, 1.0, 1.0)
    q16: np.ndarray | None = None
    k16: np.ndarray | None = None
    v16: np.ndarray | None = None
    meta: dict = field(default_factory=dict)


def fp32_qkv(wl: Workload, seed: int = SEED):
    """The float32 Q, K, V of a workload (BSHD)."""
    sq, sk, sv = wl.shapes()
    q = normal(sq, seed, STREAM_Q)
    k = normal(sk, seed, STREAM_K)
    v = normal(sv, seed, STREAM_V)
    meta = {}
    if wl.kind == "activation":
        q, k, meta = _activation_like(wl, q, k, seed)
    elif wl.kind == "sink":
        q, k, meta = _sink(wl, q, k)
    elif wl.kind == "kbias":
        k, meta = _kbias(wl, k, seed)
    elif wl.kind in FIG15_KINDS:
        q, k, v, meta = _fig15(wl, q, k, v, seed)
    elif wl.kind == "far_blocks":
        q, k, meta = _sink(wl, q, k)
        v = v + np.float32(FAR_BLOCKS_V_MEAN)
        meta["v_mean"] = FAR_BLOCKS_V_MEAN
    elif wl.kind != "gaussian":
        raise ValueError(f"unknown input kind {wl.kind!r}")
    return q, k, v, meta


def make_inputs(wl: Workload, seed: int = SEED, fp8: bool = True,
                bf16: bool = False) -> Inputs:
    q, k, v, meta = fp32_qkv(wl, seed)
    inp = Inputs(wl, meta=meta)
    if fp8:
        inp.q8, dq = quantize_e4m3(q)
        inp.k8, dk = quantize_e4m3(k)
        inp.v8, dv = quantize_e4m3(v)
        inp.descale = (dq, dk, dv)
    if bf16:
        inp.q16, inp.k16, inp.v16 = to_bf16_bits(q), to_bf16_bits(k), to_bf16_bits(v)
    return inp


def sample_rows(wl: Workload, per_head: int = 512, seed: int = ROW_SAMPLE_SEED,
                heads=None) -> np.ndarray:
    """Flat row ids (b*Hq + h)*N + i: all rows when N <= per_head, else rows
    0, N-1, the tile edges 127/128/255/256 and uniform others, per (b, h)."""
    rng = np.random.default_rng(seed)
    N = wl.N
    if N <= per_head:
        local = np.arange(N)
    else:
        fixed = [r for r in (0, 127, 128, 255, 256, N - 1) if r < N]
        rest = rng.choice(np.setdiff1d(np.arange(N), fixed),
                          per_head - len(fixed), replace=False)
        local = np.sort(np.concatenate([fixed, rest]))
    bh = np.arange(wl.B * wl.Hq) if heads is None else np.asarray(heads)
    return (bh[:, None] * N + local[None, :]).reshape(-1).astype(np.int64)


# --------------------------------------------------------------------------
# activation-like inputs
# --------------------------------------------------------------------------
OUTLIER_CHANNELS = 4
OUTLIER_GAIN = 20.0
TARGET_FAR_SHARE = 0.90      # share of (row, 64-key block) pairs > 8 binades down


def _far_share(q, k, wl: Workload, alpha: float, rows, far: float = 8.0):
    """Share of visible (row, 64-key block) pairs whose block maximum of the
    base-2 score lies more than ``far`` binades below the row maximum."""
    c = np.log2(np.e) / np.sqrt(wl.d_qk)
    grp = wl.Hq // wl.Hkv
    hits = tot = 0
    for b, h, i in rows:
        s = (k[b, :i + 1, h // grp, :].astype(np.float64)
             @ q[b, i, h, :].astype(np.float64)) * (c * alpha)
        nb = (i + 64) // 64
        pad = np.full(nb * 64, -np.inf)
        pad[:i + 1] = s
        bm = pad.reshape(nb, 64).max(axis=1)
        gap = s.max() - bm
        hits += int(np.sum(gap > far))
        tot += nb
    return hits / max(tot, 1)


def _activation_like(wl: Workload, q, k, seed: int):
    """Q, K with OUTLIER_CHANNELS channels per KV head scaled by OUTLIER_GAIN,
    then Q scaled by alpha, found by bisection so that about 90% of visible
    (row, 64-key block) pairs sit more than 8 binades below the row max."""
    rng = np.random.default_rng(seed + 77)
    grp = wl.Hq // wl.Hkv
    for g in range(wl.Hkv):
        ch = rng.choice(wl.d_qk, OUTLIER_CHANNELS, replace=False)
        k[:, :, g, ch] *= OUTLIER_GAIN
        for h in range(g * grp, (g + 1) * grp):
            q[:, :, h, ch] *= OUTLIER_GAIN
    srng = np.random.default_rng(seed + 78)
    rows = [(int(srng.integers(wl.B)), int(srng.integers(wl.Hq)),
             int(srng.integers(wl.N // 4, wl.N))) for _ in range(48)]
    lo, hi = -12.0, 6.0                   # log2(alpha) bracket
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        if _far_share(q, k, wl, 2.0 ** mid, rows) < TARGET_FAR_SHARE:
            lo = mid
        else:
            hi = mid
    alpha = float(2.0 ** (0.5 * (lo + hi)))
    q *= np.float32(alpha)
    meta = {
        "alpha": alpha,
        "far8_share": _far_share(q, k, wl, 1.0, rows, 8.0),
        "far16_share": _far_share(q, k, wl, 1.0, rows, 16.0),
    }
    return q, k, meta


# --------------------------------------------------------------------------
# sink inputs
# --------------------------------------------------------------------------
SINK_GAP = 14.0              # base-2 score of the sink key above the Gaussian part


def _sink(wl: Workload, q, k, gap: float = SINK_GAP):
    """Key 0 of every (batch, KV head) is a sink: channel 0 of every query is
    4 and channel 0 of key 0 is set so that the sink's base-2 score sits about
    ``gap`` above the rest; channel 0 of the other keys is 0.  Every later
    64-key block then lies roughly gap - 2 ... gap binades below the row
    maximum, with a per-row spread."""
    c = np.log2(np.e) / np.sqrt(wl.d_qk)
    q[..., 0] = 4.0
    k[:, :, :, 0] = 0.0
    k[:, 0, :, 0] = np.float32(gap / (c * 4.0))
    return q, k, {"sink_gap": gap}


# Blocks far below the row maximum that still carry mass, and values with a
# common direction (real value vectors have non-zero means): the pattern of
# Fig. 5, where probabilities lost to rounding bias the output instead of
# averaging out.
FAR_BLOCKS_V_MEAN = 1.0


# --------------------------------------------------------------------------
# keys with a shared offset
# --------------------------------------------------------------------------
KBIAS_STREAM = 3
KBIAS_SCALE = 4.0           # per-channel offset ~ N(0, KBIAS_SCALE^2)


def _kbias(wl: Workload, k, seed: int):
    """Every key of KV head g gets the same offset vector bias[b, g, :],
    drawn from N(0, KBIAS_SCALE^2): the keys then have a large mean over the
    sequence, which K smoothing removes."""
    bias = normal((wl.B, 1, wl.Hkv, wl.d_qk), seed, KBIAS_STREAM) * np.float32(KBIAS_SCALE)
    return k + bias, {"kbias_scale": KBIAS_SCALE}


# --------------------------------------------------------------------------
# the synthetic accuracy inputs of Fig. 15 ("ZYFA: Speed and Accuracy of FP8
# FlashAttention on AMD CDNA4", Sec. VI, Fig. 15), from their descriptions
# --------------------------------------------------------------------------
FIG15_KINDS = ("f15_gaussian", "logit_sd1", "logit_sd4", "logit_sd16", "stepped_max", "sink4",
               "rising", "alternating", "sink_flat", "full_range")
F15_SIGMA = 0.1              # Gaussian: q, k, v ~ N(0, 0.1^2)
F15_STEP_NATS = 1.0          # Stepped Max: logit step per 64-key block (not printed)
F15_RAMP_NATS = 16.0         # Rising / Alternating: total rise over the keys (not printed)
F15_SINK_NATS = 12.0         # Sink + Flat Tail: first key above the rest
F15_FLAT_SD = 0.1            # Sink + Flat Tail: logit SD of the "nearly uniform" rest
F15_SINK4_GAIN = 8.0         # 4-Key Sink: the first four keys scaled by 8
F15_RANGE = (-6.0, 8.0)      # Full Range: log2 of the magnitude, uniform
F15_CH_GAIN = 4.0            # value of the query channel that carries a key-side offset
STREAM_F15_U = 4             # streams 4, 5, 6: the uniforms of q, k, v (Full Range)


def _logit_offset(wl: Workload, q, k, ch: int, per_key, rows=None):
    """Add per_key[j] nats to the logit q_i . k_j / sqrt(d_qk) of every query
    row i (or of the rows selected by the boolean ``rows`` mask) through one
    channel: q[..., ch] = F15_CH_GAIN there (0 elsewhere) and k[:, j, :, ch] =
    per_key[j] sqrt(d_qk) / F15_CH_GAIN."""
    q[..., ch] = np.float32(F15_CH_GAIN)
    if rows is not None:
        q[:, ~rows, :, ch] = 0.0
    k[:, :, :, ch] = (np.asarray(per_key, dtype=np.float64) * np.sqrt(wl.d_qk)
                      / F15_CH_GAIN).astype(np.float32)[None, :, None]


def _uniform(shape, seed: int, stream: int) -> np.ndarray:
    """Uniform (0, 1) values as the normal CDF of the stream's N(0, 1) draws."""
    from scipy.special import ndtr
    return ndtr(normal(shape, seed, stream).astype(np.float64))


def _fig15(wl: Workload, q, k, v, seed: int):
    """Fig. 15's inputs from their descriptions, on standard normal q, k, v
    (where the figure leaves a size open the constant above is this
    module's reading):
      f15_gaussian   q, k, v ~ N(0, 0.1^2) (the timing runs' draw);
      logit_sd{1,4,16}  q and k scaled by 1, 2, 4: logits with SD 1, 4, 16 nats;
      stepped_max    each successive 64-key block F15_STEP_NATS higher;
      sink4          the first four keys scaled by 8;
      rising         a linear ramp along the keys, F15_RAMP_NATS over N keys;
      alternating    the same ramp on every other query row (even rows);
      sink_flat      q, k scaled to a logit SD of F15_FLAT_SD, key 0 raised
                     F15_SINK_NATS above them;
      full_range     every element of q, k, v: a random sign times 2^u, u
                     uniform in [-6, 8]."""
    kind = wl.kind
    N = wl.N
    j = np.arange(N, dtype=np.float64)
    meta = {"fig15": kind}
    if kind == "f15_gaussian":
        q, k, v = (x * np.float32(F15_SIGMA) for x in (q, k, v))
    elif kind.startswith("logit_sd"):
        g = np.float32(np.sqrt(float(kind[len("logit_sd"):])))
        q, k = q * g, k * g
    elif kind == "stepped_max":
        _logit_offset(wl, q, k, 0, F15_STEP_NATS * (j // 64))
    elif kind == "sink4":
        k[:, :4] *= np.float32(F15_SINK4_GAIN)
    elif kind in ("rising", "alternating"):
        rows = (np.arange(N) % 2 == 0) if kind == "alternating" else None
        _logit_offset(wl, q, k, 0, F15_RAMP_NATS * j / N, rows)
    elif kind == "sink_flat":
        g = np.float32(np.sqrt(F15_FLAT_SD))
        q, k = q * g, k * g
        _logit_offset(wl, q, k, 0, np.where(j == 0, F15_SINK_NATS, 0.0))
    elif kind == "full_range":
        lo, hi = F15_RANGE
        out = []
        for t, x in enumerate((q, k, v)):
            u = _uniform(x.shape, seed, STREAM_F15_U + t)
            mag = np.exp2(lo + (hi - lo) * u)
            out.append((np.sign(x) * mag).astype(np.float32))
        q, k, v = out
    return q, k, v, meta
