"""GB300 (sm_103a) causal attention forward: FP8 e4m3 with Lean P / exact P,
per-64-key power-of-two block scaling and division by the sum of the rounded
probabilities, and the BF16 path beside it.

This module is the thin Python binding of ``libzyfa.so`` (C ABI declared in
``include/zyfa.h``).  It only marshals arguments: every step of the
computation runs in the library's CUDA kernels.  PyTorch is used for device
memory and streams.  There is no CPU fallback: when the library has not been
built, importing the binding's functions raises.

Method: "ZYFA: Speed and Accuracy of FP8 FlashAttention on AMD CDNA4"
(Sec. II-B, II-C, IV-A, IV-B).
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB_PATH, build  # noqa: F401

ZYFA_OK = 0
ZYFA_ERR_NULL = -1
ZYFA_ERR_SHAPE = -2
ZYFA_ERR_UNSUPPORTED = -3
ZYFA_ERR_ALIGN = -4
ZYFA_ERR_CUDA = -5
ZYFA_ERR_TIMEOUT = -6
ZYFA_ERR_SCRATCH = -7
ZYFA_P_EXACT = 0
ZYFA_P_LEAN = 1

EXPORTS = ("zyfa_fwd", "zyfa_fwd_bf16", "zyfa_fwd_ex", "zyfa_fwd_bf16_ex",
           "zyfa_fwd_strided", "zyfa_fwd_bf16_strided", "zyfa_fwd_bf16qk_fp8pv",
           "zyfa_fwd_partial", "zyfa_fwd_bf16_partial", "zyfa_merge",
           "zyfa_fwd_host", "zyfa_fwd_host_workspace_bytes", "zyfa_fwd_host_plan",
           "zyfa_quantize", "zyfa_quantize_noalloc", "zyfa_status_string", "zyfa_last_device_status", "zyfa_selftest_timeout",
           "zyfa_version")

_lib = None


class ZyfaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {zyfa_status_string(status)} (status {status})")


def load():
    """Load libzyfa.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: the CUDA library must be built first "
            "(fp8_causal_flashattention_gb300.build() or __graft_entry__.build())")
    lib = ctypes.CDLL(LIB_PATH)
    vp, ci = ctypes.c_void_p, ctypes.c_int
    lib.zyfa_fwd.restype = ci
    lib.zyfa_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp] + [ci] * 9 + [vp]
    lib.zyfa_fwd_bf16.restype = ci
    lib.zyfa_fwd_bf16.argtypes = [vp, vp, vp, vp] + [ci] * 7 + [vp]
    lib.zyfa_fwd_ex.restype = ci
    lib.zyfa_fwd_ex.argtypes = [vp] * 8 + [ci] * 9 + [vp]
    lib.zyfa_fwd_bf16_ex.restype = ci
    lib.zyfa_fwd_bf16_ex.argtypes = [vp] * 5 + [ci] * 7 + [vp]
    lib.zyfa_fwd_strided.restype = ci
    lib.zyfa_fwd_strided.argtypes = [vp] * 8 + [ci] * 9 + [vp, vp]
    lib.zyfa_fwd_bf16_strided.restype = ci
    lib.zyfa_fwd_bf16_strided.argtypes = [vp] * 5 + [ci] * 7 + [vp, vp]
    lib.zyfa_fwd_bf16qk_fp8pv.restype = ci
    lib.zyfa_fwd_bf16qk_fp8pv.argtypes = [vp] * 6 + [ci] * 9 + [vp, vp]
    lib.zyfa_quantize.restype = ci
    lib.zyfa_fwd_partial.argtypes = [vp] * 8 + [ci] * 11 + [vp, vp]
    lib.zyfa_fwd_partial.restype = ci
    lib.zyfa_fwd_bf16_partial.argtypes = [vp] * 5 + [ci] * 9 + [vp, vp]
    lib.zyfa_fwd_bf16_partial.restype = ci
    lib.zyfa_merge.argtypes = [vp, vp, ci, vp, vp] + [ci] * 4 + [vp]
    lib.zyfa_merge.restype = ci
    lib.zyfa_fwd_host.argtypes = [vp] * 6 + [ci] * 10 + [vp, ctypes.c_size_t, vp]
    lib.zyfa_fwd_host.restype = ci
    lib.zyfa_fwd_host_workspace_bytes.argtypes = [ci] * 7
    lib.zyfa_fwd_host_workspace_bytes.restype = ctypes.c_size_t
    lib.zyfa_fwd_host_plan.argtypes = [ci] * 4 + [vp, ci]
    lib.zyfa_fwd_host_plan.restype = ci
    lib.zyfa_quantize.argtypes = [vp, vp, ci, ctypes.c_float, vp, vp, vp] + [ci] * 4 + [vp]
    lib.zyfa_quantize_noalloc.restype = ci
    lib.zyfa_quantize_noalloc.argtypes = lib.zyfa_quantize.argtypes
    lib.zyfa_status_string.restype = ctypes.c_char_p
    lib.zyfa_status_string.argtypes = [ci]
    lib.zyfa_last_device_status.restype = ci
    lib.zyfa_last_device_status.argtypes = [vp]
    lib.zyfa_selftest_timeout.restype = ci
    lib.zyfa_selftest_timeout.argtypes = [vp]
    lib.zyfa_version.restype = ci
    lib.zyfa_version.argtypes = []
    _lib = lib
    return lib


def _ptr(x):
    """Address of a tensor's data (or an int / None passed through)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------- C ABI, 1:1
def zyfa_fwd(q, k, v, descale_q, descale_k, descale_v, out, B, Hq, Hkv, N, d_qk, d_v,
             causal=1, p_mode=ZYFA_P_LEAN, block_scale=1, stream=None) -> int:
    """``zyfa_fwd`` of include/zyfa.h; tensors or raw device addresses."""
    return load().zyfa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(descale_q), _ptr(descale_k),
                           _ptr(descale_v), _ptr(out), B, Hq, Hkv, N, d_qk, d_v, causal,
                           p_mode, block_scale, _stream(stream))


def zyfa_fwd_bf16(q, k, v, out, B, Hq, Hkv, N, d_qk, d_v, causal=1, stream=None) -> int:
    """``zyfa_fwd_bf16`` of include/zyfa.h; tensors or raw device addresses."""
    return load().zyfa_fwd_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, N, d_qk,
                                d_v, causal, _stream(stream))


def zyfa_fwd_ex(q, k, v, descale_q, descale_k, descale_v, out, lse, B, Hq, Hkv, N, d_qk, d_v,
                causal=1, p_mode=ZYFA_P_LEAN, block_scale=1, stream=None) -> int:
    """``zyfa_fwd_ex`` of include/zyfa.h (``lse`` may be None)."""
    return load().zyfa_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(descale_q), _ptr(descale_k),
                              _ptr(descale_v), _ptr(out), _ptr(lse), B, Hq, Hkv, N, d_qk, d_v,
                              causal, p_mode, block_scale, _stream(stream))


def zyfa_fwd_bf16_ex(q, k, v, out, lse, B, Hq, Hkv, N, d_qk, d_v, causal=1, stream=None) -> int:
    """``zyfa_fwd_bf16_ex`` of include/zyfa.h (``lse`` may be None)."""
    return load().zyfa_fwd_bf16_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv,
                                   N, d_qk, d_v, causal, _stream(stream))


def zyfa_quantize(x, signs, smooth, static_descale, out, descale_out, mean_out, B, N, H, D,
                  stream=None) -> int:
    """``zyfa_quantize`` of include/zyfa.h (``signs`` / ``mean_out`` may be None)."""
    return load().zyfa_quantize(_ptr(x), _ptr(signs), int(smooth), float(static_descale),
                                _ptr(out), _ptr(descale_out), _ptr(mean_out), B, N, H, D,
                                _stream(stream))


def zyfa_quantize_noalloc(x, signs, smooth, static_descale, out, descale_out, mean_out, B, N,
                          H, D, stream=None) -> int:
    """``zyfa_quantize_noalloc`` of include/zyfa.h: zyfa_quantize with its
    scratch in the library's fixed device buffer (no device allocation)."""
    return load().zyfa_quantize_noalloc(_ptr(x), _ptr(signs), int(smooth),
                                        float(static_descale), _ptr(out), _ptr(descale_out),
                                        _ptr(mean_out), B, N, H, D, _stream(stream))


def _strides_arg(strides):
    """12 int64 element strides as a ctypes array (or None)."""
    if strides is None:
        return None
    arr = (ctypes.c_longlong * 12)(*[int(x) for x in strides])
    return ctypes.cast(arr, ctypes.c_void_p), arr


def zyfa_fwd_strided(q, k, v, descale_q, descale_k, descale_v, out, lse, B, Hq, Hkv, N, d_qk,
                     d_v, causal=1, p_mode=ZYFA_P_LEAN, block_scale=1, strides=None,
                     stream=None) -> int:
    """``zyfa_fwd_strided`` of include/zyfa.h; ``strides``: 12 element strides or None."""
    sa = _strides_arg(strides)
    return load().zyfa_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(descale_q), _ptr(descale_k),
                                   _ptr(descale_v), _ptr(out), _ptr(lse), B, Hq, Hkv, N, d_qk,
                                   d_v, causal, p_mode, block_scale,
                                   None if sa is None else sa[0], _stream(stream))


def zyfa_fwd_bf16_strided(q, k, v, out, lse, B, Hq, Hkv, N, d_qk, d_v, causal=1, strides=None,
                          stream=None) -> int:
    """``zyfa_fwd_bf16_strided`` of include/zyfa.h."""
    sa = _strides_arg(strides)
    return load().zyfa_fwd_bf16_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq,
                                        Hkv, N, d_qk, d_v, causal,
                                        None if sa is None else sa[0], _stream(stream))


def zyfa_fwd_bf16qk_fp8pv(q, k, v, descale_v, out, lse, B, Hq, Hkv, N, d_qk, d_v, causal=1,
                          p_mode=ZYFA_P_LEAN, block_scale=1, strides=None, stream=None) -> int:
    """``zyfa_fwd_bf16qk_fp8pv`` of include/zyfa.h."""
    sa = _strides_arg(strides)
    return load().zyfa_fwd_bf16qk_fp8pv(_ptr(q), _ptr(k), _ptr(v), _ptr(descale_v), _ptr(out),
                                        _ptr(lse), B, Hq, Hkv, N, d_qk, d_v, causal, p_mode,
                                        block_scale, None if sa is None else sa[0],
                                        _stream(stream))


def zyfa_fwd_partial(q, k, v, descale_q, descale_k, descale_v, out, lse, B, Hq, Hkv, N, d_qk,
                     d_v, causal=1, p_mode=ZYFA_P_LEAN, block_scale=1, key_begin=0,
                     key_end=None, strides=None, stream=None) -> int:
    """``zyfa_fwd_partial`` of include/zyfa.h (``key_end`` None: N)."""
    sa = _strides_arg(strides)
    return load().zyfa_fwd_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(descale_q), _ptr(descale_k),
                                   _ptr(descale_v), _ptr(out), _ptr(lse), B, Hq, Hkv, N, d_qk,
                                   d_v, causal, p_mode, block_scale, key_begin,
                                   N if key_end is None else key_end,
                                   None if sa is None else sa[0], _stream(stream))


def zyfa_fwd_bf16_partial(q, k, v, out, lse, B, Hq, Hkv, N, d_qk, d_v, causal=1, key_begin=0,
                          key_end=None, strides=None, stream=None) -> int:
    """``zyfa_fwd_bf16_partial`` of include/zyfa.h (``key_end`` None: N)."""
    sa = _strides_arg(strides)
    return load().zyfa_fwd_bf16_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq,
                                        Hkv, N, d_qk, d_v, causal, key_begin,
                                        N if key_end is None else key_end,
                                        None if sa is None else sa[0], _stream(stream))


def zyfa_merge(outs, lses, out, lse, B, Hq, N, d_v, stream=None) -> int:
    """``zyfa_merge`` of include/zyfa.h: ``outs`` / ``lses`` are sequences of
    tensors or device addresses (marshalled into host pointer arrays)."""
    n = len(outs)
    if len(lses) != n:
        raise ValueError("outs and lses must have the same length")
    po = (ctypes.c_void_p * max(n, 1))(*[_ptr(o) for o in outs])
    pl = (ctypes.c_void_p * max(n, 1))(*[_ptr(x) for x in lses])
    return load().zyfa_merge(ctypes.cast(po, ctypes.c_void_p), ctypes.cast(pl, ctypes.c_void_p),
                             n, _ptr(out), _ptr(lse), B, Hq, N, d_v, _stream(stream))


def zyfa_fwd_host(q, k, v, descale, out, lse, B, Hq, Hkv, N, d_qk, d_v, causal=1,
                  p_mode=ZYFA_P_LEAN, block_scale=1, n_chunks=0, workspace=None,
                  workspace_bytes=0, stream=None) -> int:
    """``zyfa_fwd_host`` of include/zyfa.h: q, k, v, out, lse are HOST tensors
    (or host addresses), ``descale`` a sequence of three floats or None,
    ``workspace`` a device tensor or address."""
    ds = None if descale is None else (ctypes.c_float * 3)(*[float(x) for x in descale])
    return load().zyfa_fwd_host(_ptr(q), _ptr(k), _ptr(v),
                                None if ds is None else ctypes.cast(ds, ctypes.c_void_p),
                                _ptr(out), _ptr(lse), B, Hq, Hkv, N, d_qk, d_v, causal, p_mode,
                                block_scale, n_chunks, _ptr(workspace), workspace_bytes,
                                _stream(stream))


def zyfa_fwd_host_workspace_bytes(B, Hq, Hkv, N, d_qk, d_v, with_lse) -> int:
    return load().zyfa_fwd_host_workspace_bytes(B, Hq, Hkv, N, d_qk, d_v, 1 if with_lse else 0)


def zyfa_fwd_host_plan(B, Hq, Hkv, n_chunks=0):
    """``zyfa_fwd_host_plan`` of include/zyfa.h: the chunk list as tuples
    (b0, nb, g0, hk, h0, hq, kv), or a negative status."""
    lib = load()
    m = lib.zyfa_fwd_host_plan(B, Hq, Hkv, n_chunks, None, 0)
    if m < 0:
        return m
    buf = (ctypes.c_int * max(7 * m, 1))()
    lib.zyfa_fwd_host_plan(B, Hq, Hkv, n_chunks, ctypes.cast(buf, ctypes.c_void_p), m)
    return [tuple(buf[7 * c:7 * c + 7]) for c in range(m)]


def zyfa_status_string(status: int) -> str:
    return load().zyfa_status_string(int(status)).decode()


def zyfa_last_device_status(stream=None) -> int:
    return load().zyfa_last_device_status(_stream(stream))


def zyfa_selftest_timeout(stream=None) -> int:
    return load().zyfa_selftest_timeout(_stream(stream))


def zyfa_version() -> int:
    return load().zyfa_version()


# ---------------------------------------------------------------- conveniences
def _shape(q, k, v):
    B, N, Hq, d_qk = q.shape
    if k.shape[0] != B or k.shape[1] != N or v.shape[:3] != k.shape[:3] or k.shape[3] != d_qk:
        raise ValueError("q, k, v must be [B, N, H, d] with matching B, N, Hkv and d_qk")
    return B, N, Hq, k.shape[2], d_qk, v.shape[3]


def _layout(q, k, v, out):
    """Element strides (b, n, h) of the four [B, N, H, d] tensors, or None when
    all are contiguous BSHD.  The last dimension must be contiguous."""
    ts = (q, k, v, out)
    if all(t.is_contiguous() for t in ts):
        return None
    st = []
    for t in ts:
        if t.stride(3) != 1:
            raise ValueError("the last (channel) dimension must be contiguous")
        st += [t.stride(0), t.stride(1), t.stride(2)]
    return st


def attention_fp8(q, k, v, descale_q=None, descale_k=None, descale_v=None, *,
                  p_mode=ZYFA_P_LEAN, block_scale=1, causal=1, out=None, return_lse=False,
                  stream=None):
    """Causal FP8 attention on e4m3 tensors (torch.float8_e4m3fn or uint8),
    [B, N, H, d] with any strides (e.g. a BHSD tensor viewed with
    ``.transpose(1, 2)``) and a contiguous last dimension; descales are
    1-element float32 device tensors (or None for 1.0).
    Returns the BF16 output [B, N, Hq, d_v] (and the FP32 LSE [B, Hq, N]
    when ``return_lse``)."""
    import torch
    B, N, Hq, Hkv, d_qk, d_v = _shape(q, k, v)
    if out is None:
        out = torch.empty((B, N, Hq, d_v), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if return_lse else None
    rc = zyfa_fwd_strided(q, k, v, descale_q, descale_k, descale_v, out, lse, B, Hq, Hkv, N, d_qk,
                          d_v, causal, p_mode, block_scale, _layout(q, k, v, out), stream)
    if rc != ZYFA_OK:
        raise ZyfaError(rc, "zyfa_fwd_strided")
    return (out, lse) if return_lse else out


def host_workspace(q, k, v, *, with_lse=False, device=None):
    """A device workspace (uint8 tensor) large enough for attention_fp8_host
    on tensors shaped like q, k, v."""
    import torch
    B, N, Hq, Hkv, d_qk, d_v = _shape(q, k, v)
    n = zyfa_fwd_host_workspace_bytes(B, Hq, Hkv, N, d_qk, d_v, with_lse)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device or "cuda")


def attention_fp8_host(q, k, v, descale=None, *, p_mode=ZYFA_P_LEAN, block_scale=1, causal=1,
                       out=None, return_lse=False, lse=None, workspace=None, n_chunks=0,
                       sync=True, stream=None):
    """Causal FP8 attention on HOST tensors, end to end in one call
    (``zyfa_fwd_host``): copies in, kernels and copies out pipelined over
    chunks of batch elements or heads.  q, k, v: CPU tensors, contiguous
    BSHD, e4m3 codes (torch.float8_e4m3fn or uint8), page-locked for the
    copies to overlap; ``descale``: three floats (q, k, v) or None;
    ``workspace``: a CUDA uint8 tensor (host_workspace), or None to allocate
    one.  Returns the host BF16 output (and the FP32 LSE [B, Hq, N]); with
    ``sync=False`` they are complete only once ``stream`` has been
    synchronised."""
    import torch
    B, N, Hq, Hkv, d_qk, d_v = _shape(q, k, v)
    for t in (q, k, v):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CPU tensors")
    pin = q.is_pinned()
    if out is None:
        out = torch.empty((B, N, Hq, d_v), dtype=torch.bfloat16, pin_memory=pin)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, pin_memory=pin)
    if workspace is None:
        workspace = host_workspace(q, k, v, with_lse=lse is not None)
    nbytes = workspace.numel() * workspace.element_size()
    rc = zyfa_fwd_host(q, k, v, descale, out, lse, B, Hq, Hkv, N, d_qk, d_v, causal, p_mode,
                       block_scale, n_chunks, workspace, nbytes, stream)
    if rc != ZYFA_OK:
        raise ZyfaError(rc, "zyfa_fwd_host")
    if sync:
        if stream is None:
            torch.cuda.current_stream().synchronize()
        elif isinstance(stream, int):
            torch.cuda.synchronize()
        else:
            stream.synchronize()
    return (out, lse) if lse is not None else out


def attention_bf16(q, k, v, *, causal=1, out=None, return_lse=False, stream=None):
    """Causal BF16 attention, BSHD.  Returns the BF16 output (and the LSE)."""
    import torch
    B, N, Hq, Hkv, d_qk, d_v = _shape(q, k, v)
    if out is None:
        out = torch.empty((B, N, Hq, d_v), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if return_lse else None
    rc = zyfa_fwd_bf16_strided(q, k, v, out, lse, B, Hq, Hkv, N, d_qk, d_v, causal,
                               _layout(q, k, v, out), stream)
    if rc != ZYFA_OK:
        raise ZyfaError(rc, "zyfa_fwd_bf16_strided")
    return (out, lse) if return_lse else out


def quantize(x, signs=None, *, smooth=False, static_descale=None, out=None, descale_out=None,
             return_mean=False, stream=None):
    """BF16 tensor [B, N, H, D] -> (e4m3 codes as torch.float8_e4m3fn, descale as a
    1-element float32 device tensor[, mean [B, H, D] float32]).

    ``signs``: None (no rotation) or a float32 device tensor of D signs, the s
    of R = diag(s)(C_m kron H_{D/m}); ``smooth``: subtract each head's mean
    over the sequence first; ``static_descale``: a power of two, or None for
    a per-call scale from the maximum."""
    import torch
    if x.dim() != 4:
        raise ValueError("x must be [B, N, H, D]")
    B, N, H, D = x.shape
    if out is None:
        out = torch.empty((B, N, H, D), dtype=torch.float8_e4m3fn, device=x.device)
    if descale_out is None:
        descale_out = torch.empty(1, dtype=torch.float32, device=x.device)
    mean = (torch.empty((B, H, D), dtype=torch.float32, device=x.device)
            if return_mean else None)
    rc = zyfa_quantize(x, signs, 1 if smooth else 0,
                       0.0 if static_descale is None else static_descale, out, descale_out,
                       mean, B, N, H, D, stream)
    if rc != ZYFA_OK:
        raise ZyfaError(rc, "zyfa_quantize")
    return (out, descale_out, mean) if return_mean else (out, descale_out)


def attention_bf16qk_fp8pv(q, k, v, descale_v=None, *, p_mode=ZYFA_P_LEAN, block_scale=1,
                           causal=1, out=None, return_lse=False, stream=None):
    """BF16 Q and K, e4m3 V (torch.float8_e4m3fn or uint8): BF16 QK^T, FP8
    probabilities and PV.  Shapes and strides as attention_fp8."""
    import torch
    B, N, Hq, Hkv, d_qk, d_v = _shape(q, k, v)
    if out is None:
        out = torch.empty((B, N, Hq, d_v), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if return_lse else None
    rc = zyfa_fwd_bf16qk_fp8pv(q, k, v, descale_v, out, lse, B, Hq, Hkv, N, d_qk, d_v, causal,
                               p_mode, block_scale, _layout(q, k, v, out), stream)
    if rc != ZYFA_OK:
        raise ZyfaError(rc, "zyfa_fwd_bf16qk_fp8pv")
    return (out, lse) if return_lse else out


def attention_partial(q, k, v, descale_q=None, descale_k=None, descale_v=None, *, key_begin=0,
                      key_end=None, p_mode=ZYFA_P_LEAN, block_scale=1, causal=1, out=None,
                      lse=None, stream=None):
    """Attention over the keys [key_begin, key_end) (multiples of 128).  FP8
    when q is float8_e4m3fn / uint8 (descales as attention_fp8), BF16 when q
    is bfloat16.  Returns (out, lse); rows that see no key of the range get
    0 and -inf."""
    import torch
    B, N, Hq, Hkv, d_qk, d_v = _shape(q, k, v)
    if out is None:
        out = torch.empty((B, N, Hq, d_v), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    st = _layout(q, k, v, out)
    if q.dtype == torch.bfloat16:
        rc = zyfa_fwd_bf16_partial(q, k, v, out, lse, B, Hq, Hkv, N, d_qk, d_v, causal,
                                   key_begin, key_end, st, stream)
    else:
        rc = zyfa_fwd_partial(q, k, v, descale_q, descale_k, descale_v, out, lse, B, Hq, Hkv, N,
                              d_qk, d_v, causal, p_mode, block_scale, key_begin, key_end, st,
                              stream)
    if rc != ZYFA_OK:
        raise ZyfaError(rc, "zyfa_fwd_partial")
    return out, lse


def merge(outs, lses, *, out=None, return_lse=True, stream=None):
    """Merge partial results (BF16 [B, N, Hq, d_v] contiguous, FP32 LSE
    [B, Hq, N]) over disjoint key ranges.  Returns out (and the merged LSE)."""
    import torch
    if not outs:
        raise ValueError("nothing to merge")
    B, N, Hq, d_v = outs[0].shape
    for o, l in zip(outs, lses):
        if tuple(o.shape) != (B, N, Hq, d_v) or not o.is_contiguous() or \
                tuple(l.shape) != (B, Hq, N) or not l.is_contiguous():
            raise ValueError("parts must be contiguous [B, N, Hq, d_v] with LSE [B, Hq, N]")
    if out is None:
        out = torch.empty((B, N, Hq, d_v), dtype=torch.bfloat16, device=outs[0].device)
    lse = (torch.empty((B, Hq, N), dtype=torch.float32, device=outs[0].device)
           if return_lse else None)
    rc = zyfa_merge(outs, lses, out, lse, B, Hq, N, d_v, stream)
    if rc != ZYFA_OK:
        raise ZyfaError(rc, "zyfa_merge")
    return (out, lse) if return_lse else out
