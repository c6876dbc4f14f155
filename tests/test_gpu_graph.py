"""The forward entry points inside a CUDA graph: every call is asynchronous
on the caller's stream and makes no allocation or host synchronisation, so
a captured call replays to the same bits as an eager one (two-tile Lean P
kernel, one-tile exact P and BF16 kernels, split-key parts with their
merge)."""
import pytest

import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def _bits(t):
    import torch
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("mode", ["lean", "exact", "bf16"])
def test_forward_replays_bit_identical(mode):
    import torch
    import fp8_causal_flashattention_gb300 as Z
    wl = S.Workload("graph", 2, 8, 4, 512, 128, 128)
    fp8 = mode != "bf16"
    inp = S.make_inputs(wl, fp8=fp8, bf16=not fp8)
    (q, k, v), ds = P.to_device(inp, fp8)
    out = torch.empty((wl.B, wl.N, wl.Hq, wl.d_v), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.B, wl.Hq, wl.N), dtype=torch.float32, device="cuda")

    def call():
        if fp8:
            pm = Z.ZYFA_P_LEAN if mode == "lean" else Z.ZYFA_P_EXACT
            rc = Z.zyfa_fwd_ex(q, k, v, ds[0], ds[1], ds[2], out, lse, wl.B, wl.Hq, wl.Hkv,
                               wl.N, wl.d_qk, wl.d_v, 1, pm, 1)
        else:
            rc = Z.zyfa_fwd_bf16_ex(q, k, v, out, lse, wl.B, wl.Hq, wl.Hkv, wl.N, wl.d_qk,
                                    wl.d_v, 1)
        assert rc == Z.ZYFA_OK

    call()
    torch.cuda.synchronize()
    ref_out, ref_lse = out.clone(), lse.clone()
    out.zero_()
    lse.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(ref_out))
    assert torch.equal(_bits(lse), _bits(ref_lse))
    assert Z.zyfa_last_device_status() == Z.ZYFA_OK


def test_split_and_merge_replay_bit_identical():
    import torch
    import fp8_causal_flashattention_gb300 as Z
    wl = S.Workload("graph_split", 1, 4, 4, 768, 128, 128)
    inp = S.make_inputs(wl)
    (q, k, v), ds = P.to_device(inp)
    cut = 384
    parts = [(torch.empty((1, wl.N, wl.Hq, 128), dtype=torch.bfloat16, device="cuda"),
              torch.empty((1, wl.Hq, wl.N), dtype=torch.float32, device="cuda"))
             for _ in range(2)]
    out = torch.empty((1, wl.N, wl.Hq, 128), dtype=torch.bfloat16, device="cuda")

    def call():
        for (o, l), (a, b) in zip(parts, ((0, cut), (cut, wl.N))):
            Z.attention_partial(q, k, v, ds[0], ds[1], ds[2], key_begin=a, key_end=b, out=o,
                                lse=l)
        Z.merge([o for o, _ in parts], [l for _, l in parts], out=out, return_lse=False)

    call()
    torch.cuda.synchronize()
    ref = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(ref))
