"""Benchmark of the causal FP8 attention forward on one GB300 (per GPU rank).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload d128] [--mode lean]

One step = one causal attention forward over the whole workload (the
configuration the metric is quoted on: B=1, Hq=Hkv=32, N=32768,
d_qk=d_v=128, FP8 e4m3 with Lean P and per-64-key block scaling), inputs
resident in HBM.  Prints one JSON line (rank 0).  Throughput is the causal
FLOP count F = 2 B Hq N^2 (d_qk + d_v) / 2 ("ZYFA", Eq. 1) over the mean
device time of one launch, timed with CUDA events on the launching stream.

--impl reference times the CPU oracle (the tests' reference implementation)
on the host cores, on bounded samples of query rows of the same workload.
Multi-GPU runs are replicas: every rank runs the whole workload on its own
GPU (no collective on the data path); value = all ranks' FLOPs / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic as S  # noqa: E402

METRIC = "FP8 causal prefill attn TFLOPS (N=32K, d=128 and MLA 192/128), % of FP8 peak"
UNIT = "TFLOP/s"
FP8_OVER_BF16 = 2.0          # nominal dense FP8 / BF16 tensor ratio (4.5 / 2.25 PF)
KERNEL_SOURCES = ["fp8_causal_flashattention_gb300/csrc/fwd.cuh",
                  "fp8_causal_flashattention_gb300/csrc/fwd3.cuh",
                  "fp8_causal_flashattention_gb300/csrc/fwd4.cuh",
                  "fp8_causal_flashattention_gb300/csrc/ptx.cuh",
                  "fp8_causal_flashattention_gb300/csrc/zyfa_api.cu"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(ms: float, ws: int, device=None) -> float:
    """The slowest rank's time: every rank's step time reduced with MAX (the
    job is as fast as its slowest replica)."""
    if ws <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(flops_per_rank: float, ws: int, ms: float) -> float:
    """TFLOP/s of the whole job: the FLOPs all ranks processed over the
    slowest rank's time."""
    return flops_per_rank * ws / (ms * 1e-3) / 1e12


def row_flops(wl: S.Workload, rows) -> float:
    i = np.asarray(rows) % wl.N
    return float(np.sum(2.0 * (i + 1) * (wl.d_qk + wl.d_v)))


# --------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# --------------------------------------------------------------------------
def oracle_sample(wl: S.Workload, inp: S.Inputs, mode: str, target_s: float, seed: int):
    """Times the oracle on a random sample of rows sized for ~target_s."""
    import oracle
    from tests import parity as P
    p = P.oracle_params(wl, inp, mode)
    q, k, v = P.qkv_for(inp, mode)
    rng = np.random.default_rng(seed)
    total = wl.B * wl.Hq * wl.N
    nthreads = oracle.default_threads()
    probe = rng.choice(total, 256, replace=False)
    t0 = time.perf_counter()
    oracle.fwd(p, q, k, v, probe, nthreads)
    rate = row_flops(wl, probe) / max(time.perf_counter() - t0, 1e-6)
    n = int(np.clip(target_s * rate / (row_flops(wl, probe) / 256), 64, total))
    rows = rng.choice(total, n, replace=False)
    t0 = time.perf_counter()
    oracle.fwd(p, q, k, v, rows, nthreads)
    dt = time.perf_counter() - t0
    return row_flops(wl, rows) / dt / 1e12, {"rows": int(n), "seconds": dt, "threads": nthreads}


def run_reference(args, wl: S.Workload):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    inp = S.make_inputs(wl)
    vals = []
    info = None
    step_s = 0.25 if args.steps > 50 else 1.5
    for i in range(args.warmup + args.steps):
        v, info = oracle_sample(wl, inp, args.mode, step_s, seed=100 + i)
        if i >= args.warmup:
            vals.append(v)
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": config_dict(wl, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": info["threads"], "kind": "oracle",
                         "sample": f"each step: {info['rows']} random query rows of the workload "
                                   f"(~{step_s}s of CPU work), TFLOP/s = sum 2(i+1)(d_qk+d_v) / time"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# GPU
# --------------------------------------------------------------------------
def config_dict(wl: S.Workload, args) -> dict:
    return {"workload": f"{wl.name}: B={wl.B} Hq={wl.Hq} Hkv={wl.Hkv} N={wl.N} d_qk={wl.d_qk} "
                        f"d_v={wl.d_v} causal, FP8 e4m3 {args.mode}",
            "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "N": wl.N, "d_qk": wl.d_qk, "d_v": wl.d_v,
            "mode": args.mode, "inputs": "N(0,1) -> per-tensor e4m3 (descale amax/448)",
            "l2": "inputs larger than L2 (no flush)"}


class ClockSampler:
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus = bus_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(", ") for r in out.strip().splitlines() if r.strip()]
        if self.bus:
            mine = [r for r in rows if len(r) > 1 and r[1].lower().endswith(self.bus.lower())]
            rows = mine or rows
        if rows and len({r[0] for r in rows}) > 1:
            first = rows[0][0]
            rows = [r for r in rows if r[0] == first]
        num = lambda x: x.replace(".", "", 1).isdigit()  # noqa: E731
        sm = [float(r[2]) for r in rows if len(r) > 2 and num(r[2])]
        mx = [float(r[3]) for r in rows if len(r) > 3 and num(r[3])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows for j in range(4)
                          if len(r) > 6 + j and r[6 + j].strip() == "Active"})
        pw = [float(r[4]) for r in rows if len(r) > 4 and num(r[4])]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(sm), "power_w_max": max(pw) if pw else None}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def stored_traffic(name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(name)
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return e.get("dram_bytes_per_launch")


def time_launches(fn, steps, warmup, stream):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_ours(args, wl: S.Workload):
    import torch
    import fp8_causal_flashattention_gb300 as Z
    from tests import parity as P

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    Z.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    inp = S.make_inputs(wl)
    (q, k, v), ds = P.to_device(inp)
    out = torch.empty((wl.B, wl.N, wl.Hq, wl.d_v), dtype=torch.bfloat16, device=dev)
    p_mode = Z.ZYFA_P_LEAN if args.mode.startswith("lean") else Z.ZYFA_P_EXACT
    bs = 0 if args.mode.endswith("nobs") else 1

    def step():
        rc = Z.zyfa_fwd(q, k, v, ds[0], ds[1], ds[2], out, wl.B, wl.Hq, wl.Hkv, wl.N, wl.d_qk,
                        wl.d_v, 1, p_mode, bs, stream)
        if rc != Z.ZYFA_OK:
            raise Z.ZyfaError(rc, "zyfa_fwd")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    props = torch.cuda.get_device_properties(local)
    bus = None
    if hasattr(props, "pci_bus_id"):
        bus = "%02X:%02X.0" % (props.pci_bus_id, getattr(props, "pci_device_id", 0))
    clk = ClockSampler(bus)
    clk.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = clk.stop()
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms, ws, dev)
    status = Z.zyfa_last_device_status()
    if status != Z.ZYFA_OK:
        raise RuntimeError(f"device status {status}")
    flops = wl.causal_flops
    value = whole_job_value(flops, ws, ms)

    # end to end through the C ABI on host buffers, every step: zyfa_fwd_host
    # copies the pinned inputs in, runs the kernels and copies the output
    # back, pipelined over chunks of heads so that copies overlap kernels
    hq, hk, hv = (torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
                  for a in (inp.q8, inp.k8, inp.v8))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    ws_bytes = Z.zyfa_fwd_host_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.N, wl.d_qk, wl.d_v, 0)
    work = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def e2e_step():
        rc = Z.zyfa_fwd_host(hq, hk, hv, inp.descale, hout, None, wl.B, wl.Hq, wl.Hkv, wl.N,
                             wl.d_qk, wl.d_v, 1, p_mode, bs, args.e2e_chunks, work, ws_bytes,
                             stream)
        if rc != Z.ZYFA_OK:
            raise Z.ZyfaError(rc, "zyfa_fwd_host")

    # the same without the pipeline: whole-tensor copies, kernel, copy back
    def serial_step():
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        step()
        hout.copy_(out, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 30))
    e2e_ms = time_launches(e2e_step, e2e_steps, 3, stream)
    serial_ms = time_launches(serial_step, e2e_steps, 2, stream)
    if Z.zyfa_last_device_status() != Z.ZYFA_OK:
        raise RuntimeError("device status after the end-to-end steps")
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = hout.numel() * hout.element_size()
    del work

    peaks, peak_src = measured_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    achieved = flops / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": config_dict(wl, args),
        "pct_of_fp8_peak": 100.0 * achieved / fp8_peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": achieved / fp8_peak,
                     "traffic": stored_traffic(f"{wl.name}_{args.mode}"),
                     "peak_source": f"{peak_src}: MEASURED_PEAKS bf16_tflops (burst) x "
                                    f"{FP8_OVER_BF16} nominal FP8/BF16 ratio",
                     "algorithmic": "F = B*Hq*N^2*(d_qk+d_v) causal FLOPs per launch"},
        "e2e": {"value": flops * ws / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "call": "zyfa_fwd_host (pinned host buffers, copies pipelined over "
                        f"n_chunks={args.e2e_chunks or 16} chunks of batch elements or heads)",
                "serial_ms_per_step": serial_ms},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "kernel_hash": kernel_hash(),
    }
    del hq, hk, hv, hout
    if not args.no_extras:
        line["also"] = extras(args, P, fp8_peak, peaks["bf16_tflops"])
    if rank == 0 and not args.no_cpu_baseline:
        v_cpu, info = oracle_sample(wl, inp, args.mode, args.cpu_seconds, seed=7)
        line["cpu_baseline"] = {
            "value": v_cpu, "unit": UNIT, "cores": info["threads"], "kind": "oracle",
            "sample": f"{info['rows']} random query rows of the workload, "
                      f"{info['seconds']:.1f} s; TFLOP/s = sum 2(i+1)(d_qk+d_v) / time"}
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def extras(args, P, fp8_peak, bf16_peak):
    """The other measured points: BF16 and exact P at d=128, and the MLA shape
    (exact P, the paper's default there, and Lean P), device-timed alike, each
    over as many launches as the headline (at least 20).  The MLA shape is
    half of the metric, so its lines carry a roofline block and the clocks of
    their timed region too."""
    import torch
    res = {}
    stream = torch.cuda.current_stream()
    steps = max(20, args.steps)
    for name, mode in (("d128", "bf16"), ("d128", "exact"), ("mla", "exact"), ("mla", "lean")):
        wl = S.WORKLOADS[name]
        inp = S.make_inputs(wl, fp8=mode != "bf16", bf16=mode == "bf16")
        dev = P.to_device(inp, mode != "bf16")
        run = lambda: P.gpu_run(inp, mode, dev)
        for _ in range(3):
            run()
        clk = ClockSampler(None)
        clk.start()
        time.sleep(0.2)
        ms = time_launches(run, steps, 0, stream)
        clocks = clk.stop()
        tf = wl.causal_flops / (ms * 1e-3) / 1e12
        peak = bf16_peak if mode == "bf16" else fp8_peak
        entry = {"tflops": tf, "ms": ms, "frac_of_peak": tf / peak, "launches": steps,
                 "clocks": clocks}
        if name == "mla":
            entry["roofline"] = {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                                 "frac": tf / peak,
                                 "traffic": stored_traffic(f"{name}_{mode}"),
                                 "algorithmic": "F = B*Hq*N^2*(d_qk+d_v) causal FLOPs per launch"}
        res[f"{name}_{mode}"] = entry
        del dev, inp
        torch.cuda.empty_cache()
    # BF16 QK^T with FP8 PV (the variant the paper's conclusion recommends)
    import fp8_causal_flashattention_gb300 as Z
    wl = S.WORKLOADS["d128"]
    inp = S.make_inputs(wl, fp8=True, bf16=True)
    q16 = torch.from_numpy(inp.q16.view(np.int16)).view(torch.bfloat16).cuda()
    k16 = torch.from_numpy(inp.k16.view(np.int16)).view(torch.bfloat16).cuda()
    v8 = torch.from_numpy(inp.v8).cuda()
    dv = torch.tensor([inp.descale[2]], dtype=torch.float32, device="cuda")
    out = torch.empty((wl.B, wl.N, wl.Hq, wl.d_v), dtype=torch.bfloat16, device="cuda")
    ms = time_launches(lambda: Z.attention_bf16qk_fp8pv(q16, k16, v8, dv, out=out), steps, 3, stream)
    tf = wl.causal_flops / (ms * 1e-3) / 1e12
    # QK^T runs at the BF16 rate and PV at the FP8 rate: the peak of the mix
    # is the harmonic combination of half the FLOPs at each
    mix_peak = 1.0 / (0.5 / bf16_peak + 0.5 / fp8_peak)
    res["d128_bf16qk_fp8pv_lean"] = {"tflops": tf, "ms": ms, "frac_of_peak": tf / mix_peak,
                                     "peak": mix_peak}
    del q16, k16, v8, out, inp
    torch.cuda.empty_cache()
    # the BHSD layout (Table VI): the same kernels on strided TMA maps
    import fp8_causal_flashattention_gb300 as Z
    wl = S.WORKLOADS["d128"]
    inp = S.make_inputs(wl)
    (q, k, v), ds = P.to_device(inp)
    qs, ks, vs = (t.transpose(1, 2).contiguous().transpose(1, 2) for t in (q, k, v))
    del q, k, v, inp
    out = torch.empty((wl.B, wl.Hq, wl.N, wl.d_v), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    ms = time_launches(lambda: Z.attention_fp8(qs, ks, vs, ds[0], ds[1], ds[2], out=out), steps, 3,
                       stream)
    tf = wl.causal_flops / (ms * 1e-3) / 1e12
    res["d128_lean_bhsd"] = {"tflops": tf, "ms": ms, "frac_of_peak": tf / fp8_peak}
    del qs, ks, vs, out
    torch.cuda.empty_cache()
    res.update(split_extras(steps, fp8_peak))
    res.update(quant_extras(steps))
    return res


def split_extras(steps, fp8_peak):
    """Split-key attention on the d=128 workload (Lean P): keys [0, N/2) and
    [N/2, N) as two partial calls, then the LSE merge (Sec. IV-B3).  The
    whole step is quoted in TFLOP/s of the full causal attention; the merge
    kernel alone in GB/s against HBM, algorithmic bytes per row = n_parts x
    (2 d_v + 4) read + (2 d_v + 4) written."""
    import torch
    import fp8_causal_flashattention_gb300 as Z
    from tests import parity as P
    peaks, _ = measured_peaks()
    wl = S.WORKLOADS["d128"]
    inp = S.make_inputs(wl)
    (q, k, v), ds = P.to_device(inp)
    del inp
    shape = (wl.B, wl.N, wl.Hq, wl.d_v)
    outs = [torch.empty(shape, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    lses = [torch.empty((wl.B, wl.Hq, wl.N), dtype=torch.float32, device="cuda")
            for _ in range(2)]
    out = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.B, wl.Hq, wl.N), dtype=torch.float32, device="cuda")
    half = wl.N // 2
    stream = torch.cuda.current_stream()

    def parts():
        for i, (a, b) in enumerate(((0, half), (half, wl.N))):
            Z.attention_partial(q, k, v, ds[0], ds[1], ds[2], key_begin=a, key_end=b,
                                out=outs[i], lse=lses[i])

    def merge():
        rc = Z.zyfa_merge(outs, lses, out, lse, wl.B, wl.Hq, wl.N, wl.d_v, stream)
        if rc != Z.ZYFA_OK:
            raise Z.ZyfaError(rc, "zyfa_merge")

    def step():
        parts()
        merge()

    ms = time_launches(step, steps, 3, stream)
    ms_merge = time_launches(merge, steps, 3, stream)
    rows = wl.B * wl.Hq * wl.N
    nbytes = rows * (2 * (2 * wl.d_v + 4) + (2 * wl.d_v + 4))
    gbs = nbytes / (ms_merge * 1e-3) / 1e9
    tf = wl.causal_flops / (ms * 1e-3) / 1e12
    res = {"d128_lean_split2_merge": {"tflops": tf, "ms": ms, "frac_of_peak": tf / fp8_peak,
                                      "launches": 3},
           "merge_d128_2parts": {"ms": ms_merge, "gbs": gbs,
                                 "frac_of_hbm": gbs / peaks["hbm_gbs"], "bytes": nbytes}}
    del q, k, v, outs, lses, out, lse
    torch.cuda.empty_cache()
    return res


def quant_extras(steps):
    """The quantisation pass before the kernel on the d=128 workload's BF16
    Q, K, V (each 32 heads x 32K x 128): Q rotated, K rotated and smoothed,
    V plain; with static scales (the fused pass of Sec. V-A) and with
    per-call scales.  HBM-bound: GB/s = algorithmic bytes / device time,
    algorithmic bytes per element = 2 (read) + 1 (write) + 2 for every
    further full read the definition needs (the mean before K smoothing,
    the maximum before a per-call scale)."""
    import torch
    import fp8_causal_flashattention_gb300 as Z
    peaks, _ = measured_peaks()
    hbm = peaks["hbm_gbs"]
    wl = S.WORKLOADS["d128"]
    q, k, v, _ = S.fp32_qkv(wl)
    dev = [torch.from_numpy(S.to_bf16_bits(a).view(np.int16)).view(torch.bfloat16).cuda()
           for a in (q, k, v)]
    del q, k, v
    signs = torch.from_numpy(S.rotation_signs(wl.d_qk)).cuda()
    outs = [torch.empty(t.shape, dtype=torch.float8_e4m3fn, device="cuda") for t in dev]
    ds = [torch.empty(1, dtype=torch.float32, device="cuda") for _ in dev]
    stream = torch.cuda.current_stream()
    n = dev[0].numel()
    res = {}
    for label, static in (("static", 2.0 ** -5), ("dynamic", None)):
        plan = ((dev[0], signs, False), (dev[1], signs, True), (dev[2], None, False))

        def step():
            for (x, s, sm), o, d in zip(plan, outs, ds):
                Z.quantize(x, s, smooth=sm, static_descale=static, out=o, descale_out=d)

        ms = time_launches(step, steps, 3, stream)
        extra = 1 + (0 if static else 3)        # K's mean pass; one max pass per tensor
        nbytes = n * (3 * 3 + 2 * extra)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[f"quant_d128_qkv_{label}"] = {"ms": ms, "gbs": gbs, "frac_of_hbm": gbs / hbm,
                                          "bytes": nbytes}
    # the quantise kernel alone: Q rotated, static scale, 3 bytes per element
    ms = time_launches(lambda: Z.quantize(dev[0], signs, static_descale=2.0 ** -5, out=outs[0],
                                          descale_out=ds[0]), steps, 3, stream)
    gbs = 3 * n / (ms * 1e-3) / 1e9
    res["quant_d128_q_rot_static"] = {"ms": ms, "gbs": gbs, "frac_of_hbm": gbs / hbm,
                                      "bytes": 3 * n}
    del dev, outs
    torch.cuda.empty_cache()
    return res


def run_sweep(args):
    """Every workload x mode, device-timed; one JSON line each (for tables)."""
    import torch
    import fp8_causal_flashattention_gb300 as Z
    from tests import parity as P
    Z.load()
    torch.cuda.set_device(0)
    peaks, _ = measured_peaks()
    stream = torch.cuda.current_stream()
    for name in ("pr1", "d128", "mla", "gqa_act", "sweep_1k", "sweep_4k", "sweep_16k", "sweep_64k"):
        wl = S.WORKLOADS[name]
        for mode in ("lean", "exact", "bf16"):
            inp = S.make_inputs(wl, fp8=mode != "bf16", bf16=mode == "bf16")
            dev = P.to_device(inp, mode != "bf16")
            steps = max(5, min(200, int(2e13 / wl.causal_flops)))
            clk = ClockSampler(None)
            clk.start()
            ms = time_launches(lambda: P.gpu_run(inp, mode, dev), steps, 3, stream)
            clocks = clk.stop()
            tf = wl.causal_flops / (ms * 1e-3) / 1e12
            peak = peaks["bf16_tflops"] * (1.0 if mode == "bf16" else FP8_OVER_BF16)
            abytes = wl.B * wl.N * (wl.Hq * wl.d_qk + wl.Hkv * (wl.d_qk + wl.d_v)) * (
                2 if mode == "bf16" else 1) + wl.B * wl.N * wl.Hq * wl.d_v * 2
            hbm_roof = abytes / (ms * 1e-3) / 1e9
            # the roof at this arithmetic intensity: min(tensor peak, AI x HBM)
            roof = min(peak, wl.causal_flops / abytes * peaks["hbm_gbs"] * 1e9 / 1e12)
            print(json.dumps({"workload": name, "mode": mode, "tflops": tf, "ms": ms,
                              "frac_of_tensor_peak": tf / peak,
                              "algorithmic_GBps": hbm_roof,
                              "frac_of_hbm": hbm_roof / peaks["hbm_gbs"],
                              "roof_tflops": roof, "frac_of_roof": tf / roof,
                              "sm_mhz": clocks.get("sm_mhz"), "reasons": clocks.get("reasons")}),
                  flush=True)
            del dev, inp
            torch.cuda.empty_cache()


def run_sustained(args):
    """Sustained throughput: for the d=128 workload and the activation-like
    GQA workload (the clock depends on the data), 1 s of warm-in, then three
    back-to-back windows of at least 1 s each, CUDA-event timed, with the SM
    clock sampled during each window.  One JSON line per workload and mode:
    mean TFLOP/s, the spread over the three windows and the median clock."""
    import torch
    import fp8_causal_flashattention_gb300 as Z
    from tests import parity as P
    Z.load()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    for name in ("d128", "gqa_act"):
        wl = S.WORKLOADS[name]
        for mode in ("lean", "exact"):
            inp = S.make_inputs(wl)
            dev = P.to_device(inp, True)
            run = lambda: P.gpu_run(inp, mode, dev)
            one = time_launches(run, 3, 2, stream)           # ms per launch, to size the windows
            n = max(3, int(1000.0 / one))                     # launches per ~1 s
            time_launches(run, n, 0, stream)                  # 1 s warm-in
            wins = []
            for _ in range(3):
                clk = ClockSampler(None)
                clk.start()
                ms = time_launches(run, n, 0, stream)
                c = clk.stop()
                wins.append((wl.causal_flops / (ms * 1e-3) / 1e12, c))
            tfs = [w[0] for w in wins]
            print(json.dumps({"workload": name, "mode": mode, "windows": 3,
                              "seconds_per_window": n * one / 1000.0,
                              "tflops_mean": float(np.mean(tfs)), "tflops_min": min(tfs),
                              "tflops_max": max(tfs),
                              "sm_mhz": [w[1].get("sm_mhz") for w in wins],
                              "power_w_max": [w[1].get("power_w_max") for w in wins],
                              "reasons": sorted({r for w in wins for r in w[1].get("reasons", [])})}),
                  flush=True)
            del dev, inp
            torch.cuda.empty_cache()


def run_accuracy(args):
    """Fig. 15's measurement on this GPU: the output error of one call on
    each synthetic input at S = 8K, as relative RMS against fp64 attention on
    the same quantised inputs (sampled rows, 64 per head), for Lean P, exact
    P and BF16, next to the oracle's ablation in the style of the compared
    FP8 kernel (exact p rounded relative to the row maximum, no block
    scaling, unrounded row sum).  One JSON line per input and head size."""
    import torch
    import oracle
    import fp8_causal_flashattention_gb300 as Z
    from tests import accuracy as A
    from tests import parity as P
    Z.load()
    torch.cuda.set_device(0)
    for d in (128, 192):
        for kind in list(S.FIG15_KINDS) + ["far_blocks"]:
            wl = S.Workload(kind, 1, 8, 8, 8192, d, 128, kind=kind)
            rows = S.sample_rows(wl, per_head=64)
            line = {"input": kind, "d_qk": d, "d_v": 128, "N": wl.N, "Hq": wl.Hq,
                    "rows": int(len(rows)), "metric": "rel RMS vs fp64 on the same inputs"}
            inp = S.make_inputs(wl, fp8=True, bf16=True)
            ref8, _ = oracle.attn_fp64(P.oracle_params(wl, inp, "lean"), inp.q8, inp.k8, inp.v8,
                                       rows)
            ref16, _ = oracle.attn_fp64(P.oracle_params(wl, inp, "bf16"), inp.q16, inp.k16,
                                        inp.v16, rows)
            for mode in ("lean", "exact", "bf16"):
                out = P.gpu_run(inp, mode)
                got = P.gather_rows(out, wl, rows)
                line[mode] = A.rel_rms(got, ref16 if mode == "bf16" else ref8)
                del out
            _, ob, _ = oracle.fwd(A.ablation_params(wl, inp), inp.q8, inp.k8, inp.v8, rows)
            line["ablation"] = A.rel_rms(oracle.bf16_bits_to_f64(ob), ref8)
            line["lean_over_ablation"] = line["lean"] / line["ablation"]
            line["exact_over_ablation"] = line["exact"] / line["ablation"]
            print(json.dumps(line), flush=True)
            del inp
            torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="d128", choices=sorted(S.WORKLOADS))
    ap.add_argument("--mode", default="lean", choices=["lean", "exact", "lean_nobs", "exact_nobs"])
    ap.add_argument("--e2e-chunks", type=int, default=0,
                    help="n_chunks of the end-to-end host call (0: the library's choice)")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sweep", action="store_true",
                    help="time every workload and mode (one JSON line each)")
    ap.add_argument("--sustained", action="store_true",
                    help="sustained throughput of the d128 and GQA workloads (3 x 1 s windows)")
    ap.add_argument("--accuracy", action="store_true",
                    help="error of one call on Fig. 15's synthetic inputs (one JSON line each)")
    args = ap.parse_args()
    if args.sweep:
        run_sweep(args)
        return
    if args.accuracy:
        run_accuracy(args)
        return
    if args.sustained:
        run_sustained(args)
        return
    wl = S.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
