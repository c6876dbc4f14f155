"""Strided layouts (zyfa_fwd_strided / zyfa_fwd_bf16_strided) on the GPU.

A BHSD tensor viewed as [B, N, H, d] through transpose(1, 2), and q, k, v
sliced out of one packed [B, N, Hq + 2 Hkv, d] tensor, must give the same
output and LSE bytes as the contiguous BSHD path (same kernels, same
arithmetic; only the addresses differ) -- and so the same parity with the
oracle, which one case checks directly.
"""
import numpy as np
import pytest

import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import fp8_causal_flashattention_gb300 as Z
    Z.build()
    Z.load()
    return Z


def _run(Z, mode, q, k, v, ds, out, causal):
    if mode == "bf16":
        return Z.attention_bf16(q, k, v, causal=causal, out=out, return_lse=True)
    return Z.attention_fp8(q, k, v, ds[0], ds[1], ds[2], p_mode=Z.ZYFA_P_LEAN if mode == "lean" else Z.ZYFA_P_EXACT,
                           causal=causal, out=out, return_lse=True)


def _bhsd_view(t):
    """A contiguous BHSD copy of a BSHD tensor, viewed as [B, N, H, d]."""
    return t.transpose(1, 2).contiguous().transpose(1, 2)


CASES = [
    # B, Hq, Hkv, N, d_qk
    (1, 2, 2, 512, 128),
    (2, 4, 1, 384, 128),
    (1, 2, 1, 256, 192),
]


@pytest.mark.parametrize("causal", [1, 0])
@pytest.mark.parametrize("mode", ["lean", "exact", "bf16"])
@pytest.mark.parametrize("case", CASES, ids=["x".join(map(str, c)) for c in CASES])
def test_bhsd_equals_bshd(lib, case, mode, causal):
    import torch
    wl = S.Workload("st", *case, 128)
    inp = S.make_inputs(wl, seed=12, fp8=mode != "bf16", bf16=mode == "bf16")
    (q, k, v), ds = P.to_device(inp, mode != "bf16")
    ref, ref_lse = _run(lib, mode, q, k, v, ds, None, causal)
    qs, ks, vs = _bhsd_view(q), _bhsd_view(k), _bhsd_view(v)
    assert not qs.is_contiguous() and qs.stride(3) == 1
    out = torch.empty((wl.B, wl.Hq, wl.N, 128), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    got, lse = _run(lib, mode, qs, ks, vs, ds, out, causal)
    torch.cuda.synchronize()
    assert got.data_ptr() == out.data_ptr()
    assert torch.equal(got.contiguous(), ref)
    assert torch.equal(lse, ref_lse)


@pytest.mark.parametrize("mode", ["lean", "exact", "bf16"])
def test_packed_qkv_equals_separate(lib, mode):
    import torch
    wl = S.Workload("pk", 2, 4, 2, 256, 128, 128)
    inp = S.make_inputs(wl, seed=13, fp8=mode != "bf16", bf16=mode == "bf16")
    (q, k, v), ds = P.to_device(inp, mode != "bf16")
    ref, ref_lse = _run(lib, mode, q, k, v, ds, None, 1)
    packed = torch.cat([q, k, v], dim=2).contiguous()        # [B, N, Hq + 2 Hkv, d]
    qp, kp, vp = packed[:, :, :4], packed[:, :, 4:6], packed[:, :, 6:8]
    got, lse = _run(lib, mode, qp, kp, vp, ds, None, 1)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    assert torch.equal(lse, ref_lse)


def test_bhsd_against_oracle(lib):
    """One BHSD case straight against the oracle, every row."""
    import torch
    wl = S.Workload("bo", 1, 2, 1, 384, 128, 128)
    inp = S.make_inputs(wl, seed=14)
    (q, k, v), ds = P.to_device(inp)
    out = torch.empty((wl.B, wl.Hq, wl.N, 128), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    got = lib.attention_fp8(_bhsd_view(q), _bhsd_view(k), _bhsd_view(v), ds[0], ds[1], ds[2], out=out)
    torch.cuda.synchronize()
    rows = np.arange(wl.B * wl.Hq * wl.N)
    res = P.errors(P.gather_rows(got.contiguous(), wl, rows), inp, "lean", rows, extra=False)
    assert res["rel_l2"] <= 1e-3, res
