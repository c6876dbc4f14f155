"""zyfa_fwd_host: the FP8 forward end to end on host buffers, with the copies
in, the kernels and the copies out pipelined over chunks of batch elements
or of key/value heads.  Attention is independent per batch element and per
head (ZYFA, Sec. II-B), and each chunk runs the forward's own kernels on a
view of the same tensors, so the output and the LSE must be bit-identical to
zyfa_fwd_ex's for every chunk plan; one case also goes to the oracle."""
import numpy as np
import pytest

import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

# (B, Hq, Hkv, N, d_qk, mode, n_chunks): plans of one chunk, batch ranges,
# head groups (with and without grouped-query heads), a group count that is
# not a divisor (3 of 8 heads -> 2 groups), more chunks than heads, d_qk=192,
# and query-head sub-ranges sharing one copied K/V head
CASES = [
    (1, 8, 8, 512, 128, "lean", 0),
    (1, 8, 8, 512, 128, "lean", 3),
    (1, 8, 2, 384, 128, "exact", 8),
    (3, 4, 2, 256, 128, "lean", 2),
    (3, 4, 2, 256, 128, "lean", 5),
    (2, 4, 4, 256, 192, "exact", 1),
    (2, 4, 1, 640, 128, "lean_nobs", 4),
    (1, 2, 2, 256, 128, "exact_nobs", 32),
    # fewer K/V heads than chunks: query heads split, K and V copied once
    (1, 8, 1, 384, 128, "lean", 8),
    (1, 16, 2, 256, 128, "exact", 8),
    (2, 6, 1, 256, 192, "lean", 5),
]


def _modes(mode):
    import fp8_causal_flashattention_gb300 as Z
    return (Z.ZYFA_P_LEAN if mode.startswith("lean") else Z.ZYFA_P_EXACT,
            0 if mode.endswith("nobs") else 1)


def _device_ref(inp, mode):
    import fp8_causal_flashattention_gb300 as Z
    (q, k, v), ds = P.to_device(inp)
    pm, bs = _modes(mode)
    out, lse = Z.attention_fp8(q, k, v, ds[0], ds[1], ds[2], p_mode=pm, block_scale=bs,
                               return_lse=True)
    return out.cpu(), lse.cpu()


def _host_inputs(inp, pinned=True):
    import torch
    ts = [torch.from_numpy(np.ascontiguousarray(a)) for a in (inp.q8, inp.k8, inp.v8)]
    return [t.pin_memory() for t in ts] if pinned else ts


def _same_bits(a, b):
    import torch
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("B,Hq,Hkv,N,dqk,mode,n", CASES)
def test_host_call_bit_identical_to_device_call(B, Hq, Hkv, N, dqk, mode, n):
    import fp8_causal_flashattention_gb300 as Z
    wl = S.Workload(f"host{B}_{Hq}_{Hkv}_{N}", B, Hq, Hkv, N, dqk, 128)
    inp = S.make_inputs(wl)
    ref_out, ref_lse = _device_ref(inp, mode)
    hq, hk, hv = _host_inputs(inp)
    pm, bs = _modes(mode)
    out, lse = Z.attention_fp8_host(hq, hk, hv, inp.descale, p_mode=pm, block_scale=bs,
                                    return_lse=True, n_chunks=n)
    assert _same_bits(out, ref_out)
    assert _same_bits(lse, ref_lse)
    assert Z.zyfa_last_device_status() == Z.ZYFA_OK


def test_host_call_pageable_buffers_and_no_lse():
    import fp8_causal_flashattention_gb300 as Z
    wl = S.Workload("host_pageable", 1, 4, 2, 384, 128, 128)
    inp = S.make_inputs(wl)
    ref_out, _ = _device_ref(inp, "lean")
    hq, hk, hv = _host_inputs(inp, pinned=False)
    out = Z.attention_fp8_host(hq, hk, hv, inp.descale, n_chunks=2)
    assert not out.is_pinned()
    assert _same_bits(out, ref_out)


def test_host_call_without_descale_is_scale_one():
    import torch
    import fp8_causal_flashattention_gb300 as Z
    wl = S.Workload("host_nodescale", 1, 4, 4, 256, 128, 128)
    inp = S.make_inputs(wl)
    (q, k, v), _ = P.to_device(inp)
    ref = Z.attention_fp8(q, k, v).cpu()
    hq, hk, hv = _host_inputs(inp)
    out = Z.attention_fp8_host(hq, hk, hv, None, n_chunks=4)
    assert _same_bits(out, ref)
    assert torch.isfinite(out.float()).all()


def test_host_call_matches_oracle():
    import fp8_causal_flashattention_gb300 as Z
    wl = S.Workload("host_oracle", 2, 4, 2, 384, 128, 128)
    inp = S.make_inputs(wl)
    hq, hk, hv = _host_inputs(inp)
    out = Z.attention_fp8_host(hq, hk, hv, inp.descale, n_chunks=4)
    rows = np.arange(wl.B * wl.Hq * wl.N)
    res = P.errors(P.gather_rows(out, wl, rows), inp, "lean", rows, extra=False)
    assert P.passes(res, "lean"), res


def test_host_call_reuses_workspace_and_orders_on_stream():
    """Back-to-back calls on one stream with one workspace: each call's
    copies in wait for the previous call's copies out."""
    import torch
    import fp8_causal_flashattention_gb300 as Z
    outs, refs = [], []
    ws = None
    for seed in (0, 1, 2):
        wl = S.Workload("host_reuse", 1, 8, 4, 512, 128, 128)
        inp = S.make_inputs(wl, seed=seed)
        refs.append(_device_ref(inp, "lean")[0])
        hq, hk, hv = _host_inputs(inp)
        if ws is None:
            ws = Z.host_workspace(hq, hk, hv)
        outs.append(Z.attention_fp8_host(hq, hk, hv, inp.descale, workspace=ws, n_chunks=4,
                                         sync=False))
    torch.cuda.synchronize()
    for o, r in zip(outs, refs):
        assert _same_bits(o, r)


def test_host_call_captured_in_cuda_graph():
    import torch
    import fp8_causal_flashattention_gb300 as Z
    wl = S.Workload("host_graph", 1, 8, 8, 512, 128, 128)
    inp = S.make_inputs(wl)
    ref_out, ref_lse = _device_ref(inp, "lean")
    hq, hk, hv = _host_inputs(inp)
    ws = Z.host_workspace(hq, hk, hv, with_lse=True)
    out = torch.empty(ref_out.shape, dtype=torch.bfloat16).pin_memory()
    lse = torch.empty(ref_lse.shape, dtype=torch.float32).pin_memory()
    kw = dict(out=out, lse=lse, workspace=ws, n_chunks=4)
    Z.attention_fp8_host(hq, hk, hv, inp.descale, **kw)          # creates the lanes
    out.zero_()
    lse.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        Z.attention_fp8_host(hq, hk, hv, inp.descale, sync=False, **kw)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert _same_bits(out, ref_out)
    assert _same_bits(lse, ref_lse)
