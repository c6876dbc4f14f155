"""Shared helpers of the GPU parity tests, smoke() and bench.py's checks.

Runs the CUDA path through the C ABI (via the thin binding) and the CPU
oracle on the same seeded inputs, and reports the errors:

* ``rel_l2`` / ``max_abs`` against the oracle's definition with the running
  maximum of the kernel (blocks of 128 keys in ascending order, lazy
  threshold tau) -- the parity gate;
* ``rel_l2_exactmax`` against the oracle with the exact row maximum (the
  paper's P-term emulation, Sec. V-E);
* ``rel_l2_fp64`` against fp64 softmax attention on the same quantised inputs
  (Sec. V-D), reported for every mode;
* ``snr_db`` against the running-maximum oracle (the paper's 30 dB gate,
  Sec. V-A).

Gates: FP8 rel-L2 <= 1e-2 and max-abs <= 3e-2 max|V|; BF16
rel-L2 <= 5e-3.
"""
from __future__ import annotations

import numpy as np

import synthetic as S

FP8_REL_L2 = 1e-2
FP8_MAX_ABS_FRAC = 3e-2
BF16_REL_L2 = 5e-3


def to_device(inp: S.Inputs, fp8: bool = True):
    import torch
    dev = torch.device("cuda", 0)
    if fp8:
        t = [torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in (inp.q8, inp.k8, inp.v8)]
        ds = [torch.tensor([d], dtype=torch.float32, device=dev) for d in inp.descale]
        return t, ds
    t = [torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
         for a in (inp.q16, inp.k16, inp.v16)]
    return t, None


def gpu_run(inp: S.Inputs, mode: str, dev_tensors=None, causal: int = 1):
    """mode: 'lean', 'exact', 'lean_nobs', 'exact_nobs' or 'bf16'.
    Returns the BF16 output as a torch tensor on the device."""
    import fp8_causal_flashattention_gb300 as Z
    fp8 = mode != "bf16"
    (q, k, v), ds = dev_tensors if dev_tensors is not None else to_device(inp, fp8)
    if not fp8:
        return Z.attention_bf16(q, k, v, causal=causal)
    p_mode = Z.ZYFA_P_LEAN if mode.startswith("lean") else Z.ZYFA_P_EXACT
    bs = 0 if mode.endswith("nobs") else 1
    return Z.attention_fp8(q, k, v, ds[0], ds[1], ds[2], p_mode=p_mode, block_scale=bs,
                           causal=causal)


def gather_rows(out, wl: S.Workload, rows) -> np.ndarray:
    """Rows (flat (b*Hq + h)*N + i) of a BSHD output as float64 [R, d_v]."""
    import torch
    rows = np.asarray(rows, dtype=np.int64)
    b = rows // (wl.Hq * wl.N)
    h = (rows // wl.N) % wl.Hq
    i = rows % wl.N
    idx = torch.from_numpy((b * wl.N + i) * wl.Hq + h).to(out.device)
    sel = out.reshape(-1, wl.d_v).index_select(0, idx)
    return sel.float().cpu().numpy().astype(np.float64)


def oracle_params(wl: S.Workload, inp: S.Inputs, mode: str, max_mode=None, causal: int = 1,
                  **extra):
    """Oracle parameters of a GPU mode; ``extra`` (e.g. key_begin / key_end)
    passes through to oracle.make_params."""
    import oracle
    if max_mode is None:
        max_mode = oracle.MAX_RUNNING
    fp8 = mode != "bf16"
    kw = dict(dtype="e4m3" if fp8 else "bf16", B=wl.B, Hq=wl.Hq, Hkv=wl.Hkv, N=wl.N,
              d_qk=wl.d_qk, d_v=wl.d_v, max_mode=max_mode, causal=causal)
    if fp8:
        kw.update(descale=inp.descale,
                  p_mode=oracle.P_LEAN if mode.startswith("lean") else oracle.P_EXACT,
                  block_scale=0 if mode.endswith("nobs") else 1)
    kw.update(extra)
    return oracle.make_params(**kw)


def qkv_for(inp: S.Inputs, mode: str):
    if mode == "bf16":
        return inp.q16, inp.k16, inp.v16
    return inp.q8, inp.k8, inp.v8


def errors(gpu_rows: np.ndarray, inp: S.Inputs, mode: str, rows, extra: bool = True,
           causal: int = 1) -> dict:
    import oracle
    wl = inp.wl
    q, k, v = qkv_for(inp, mode)
    p = oracle_params(wl, inp, mode, causal=causal)
    ref, ref_bf16, _ = oracle.fwd(p, q, k, v, rows)
    ref_b = oracle.bf16_bits_to_f64(ref_bf16)
    diff = gpu_rows - ref_b
    res = {
        "rows": int(len(rows)),
        "rel_l2": float(np.linalg.norm(diff) / np.linalg.norm(ref_b)),
        "max_abs": float(np.max(np.abs(diff))),
        "nonfinite": int(np.sum(~np.isfinite(gpu_rows))),
        "snr_db": float(10 * np.log10(np.sum(ref_b ** 2) / max(np.sum(diff ** 2), 1e-300))),
    }
    if mode == "bf16":
        vmax = float(np.max(np.abs(oracle.bf16_bits_to_f64(inp.v16))))
    else:
        vmax = float(np.max(np.abs(oracle.e4m3_decode_table()[inp.v8]))) * inp.descale[2]
    res["max_abs_frac"] = res["max_abs"] / vmax
    if extra:
        pe = oracle_params(wl, inp, mode, max_mode=oracle.MAX_EXACT, causal=causal)
        refe, _, _ = oracle.fwd(pe, q, k, v, rows)
        ref64, _ = oracle.attn_fp64(p, q, k, v, rows)
        res["rel_l2_exactmax"] = float(np.linalg.norm(gpu_rows - refe) / np.linalg.norm(refe))
        res["rel_l2_fp64"] = float(np.linalg.norm(gpu_rows - ref64) / np.linalg.norm(ref64))
        res["oracle_rel_l2_fp64"] = float(np.linalg.norm(ref - ref64) / np.linalg.norm(ref64))
        # the oracle's output rounded to BF16 as the kernels' (the like-for-like distance)
        res["oracle_bf16_rel_l2_fp64"] = float(np.linalg.norm(ref_b - ref64) /
                                               np.linalg.norm(ref64))
    return res


def passes(res: dict, mode: str) -> bool:
    if res["nonfinite"]:
        return False
    if mode == "bf16":
        return res["rel_l2"] <= BF16_REL_L2
    return res["rel_l2"] <= FP8_REL_L2 and res["max_abs_frac"] <= FP8_MAX_ABS_FRAC
