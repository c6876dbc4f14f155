"""Tensors addressed past 2^32 bytes.  The paper's kernels keep 32-bit
offsets and fall back to a slower kernel beyond them; here the tensor maps
take 64-bit strides with per-dimension coordinates and the epilogue forms
64-bit addresses, so one kernel serves every size.  Each batch element of
q, k, v and out is placed 4 GiB + 1 MiB after the previous one (through the
strided entry points) and the result must be bit-identical to the same
problem in contiguous tensors."""
import pytest

import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

GAP = (1 << 32) + (1 << 20)          # bytes from one batch element to the next


def _spread(x):
    """A copy of x [B, N, H, d] whose batch elements sit GAP bytes apart."""
    import torch
    B, N, H, d = x.shape
    esz = x.element_size()
    buf = torch.empty((B - 1) * GAP + N * H * d * esz, dtype=torch.uint8, device=x.device)
    y = torch.as_strided(buf.view(x.dtype), (B, N, H, d), (GAP // esz, H * d, d, 1))
    y.copy_(x)
    return y, buf


def _bits(t):
    import torch
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("mode,dqk", [("lean", 128), ("exact", 128), ("lean", 192), ("bf16", 128)])
def test_batches_past_4gib_bit_identical(mode, dqk):
    import torch
    import fp8_causal_flashattention_gb300 as Z
    wl = S.Workload("far", 2, 2, 2, 256, dqk, 128)
    fp8 = mode != "bf16"
    inp = S.make_inputs(wl, fp8=fp8, bf16=not fp8)
    (q, k, v), ds = P.to_device(inp, fp8)
    pm = Z.ZYFA_P_LEAN if mode == "lean" else Z.ZYFA_P_EXACT
    if fp8:
        ref, ref_lse = Z.attention_fp8(q, k, v, ds[0], ds[1], ds[2], p_mode=pm, return_lse=True)
    else:
        ref, ref_lse = Z.attention_bf16(q, k, v, return_lse=True)
    bufs = []
    qf, b = _spread(q); bufs.append(b)
    kf, b = _spread(k); bufs.append(b)
    vf, b = _spread(v); bufs.append(b)
    of, b = _spread(torch.zeros_like(ref)); bufs.append(b)
    assert qf.stride(0) * qf.element_size() > (1 << 32)
    if fp8:
        out, lse = Z.attention_fp8(qf, kf, vf, ds[0], ds[1], ds[2], p_mode=pm, out=of,
                                   return_lse=True)
    else:
        out, lse = Z.attention_bf16(qf, kf, vf, out=of, return_lse=True)
    torch.cuda.synchronize()
    assert Z.zyfa_last_device_status() == Z.ZYFA_OK
    assert out.data_ptr() == of.data_ptr()
    assert torch.equal(_bits(out.contiguous()), _bits(ref))
    assert torch.equal(_bits(lse), _bits(ref_lse))
    del qf, kf, vf, of, out, bufs
    torch.cuda.empty_cache()
