"""zyfa_quantize_noalloc against zyfa_quantize (GPU).

The no-alloc entry point runs the same kernels with its scratch in a fixed
device array, so on the same inputs its outputs must equal zyfa_quantize's
bit for bit -- on two calls in a row, which also shows that nothing left in
the shared array by one call leaks into the next.  The default device
memory pool's high-water mark shows that it allocates nothing while
zyfa_quantize does.  This file is named to be collected last; it passes
alone and after the other GPU tests.
"""
import ctypes
import os

import numpy as np
import pytest

import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import fp8_causal_flashattention_gb300 as Z
    Z.build()
    Z.load()
    return Z


def _bf16(shape, seed, kbias):
    x = S.normal(shape, seed, 30)
    if kbias:
        x = x + S.normal((shape[0], 1, shape[2], shape[3]), seed, 31) * np.float32(4.0)
    return S.to_bf16_bits(x)


def _run(lib, fn, x, signs, smooth, static, with_mean):
    import torch
    B, N, H, D = x.shape
    out = torch.full((B, N, H, D), 0x55, dtype=torch.uint8, device="cuda")
    d = torch.full((1,), -3.0, device="cuda")
    mean = torch.full((B, H, D), 7.0, device="cuda") if with_mean else None
    rc = fn(x, signs, int(smooth), 0.0 if static is None else static, out, d, mean, B, N, H, D)
    assert rc == lib.ZYFA_OK, lib.zyfa_status_string(rc)
    torch.cuda.synchronize()
    return out.cpu(), d.cpu(), None if mean is None else mean.cpu()


CASES = [
    # shape, rotate, smooth, static descale, mean_out
    ((1, 32768, 32, 128), True, True, None, False),     # K of the N = 32K, 32-head prefill
    ((2, 1000, 8, 128), True, True, None, True),
    ((1, 333, 4, 192), True, True, 2.0 ** -3, False),
    ((3, 64, 5, 192), False, True, None, True),
    ((2, 100, 3, 128), True, False, None, False),       # per-call scale only
    ((1, 7, 3, 128), False, False, 0.5, False),         # no scratch at all
]


@pytest.mark.parametrize("case", CASES, ids=[f"{'x'.join(map(str, c[0]))}-{i}" for i, c in enumerate(CASES)])
def test_noalloc_matches_allocating_entry_point_twice(lib, case):
    import torch
    shape, rot, smooth, static, with_mean = case
    x = torch.from_numpy(_bf16(shape, sum(shape), smooth).view(np.int16)).view(torch.bfloat16).cuda()
    signs = torch.from_numpy(S.rotation_signs(shape[3])).cuda() if rot else None
    ref = _run(lib, lib.zyfa_quantize, x, signs, smooth, static, with_mean)
    for _ in range(2):
        got = _run(lib, lib.zyfa_quantize_noalloc, x, signs, smooth, static, with_mean)
        assert torch.equal(got[0], ref[0])
        assert torch.equal(got[1], ref[1])
        if with_mean:
            assert torch.equal(got[2], ref[2])


def _default_pool_used_high():
    """(current, reset, read_high) of the device default memory pool: the
    memory in use now, the reset of the used-memory high water mark (which
    sets it to the memory in use) and its value, through the CUDA runtime
    library."""
    for name in ("libcudart.so.13", "libcudart.so",
                 os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64", "libcudart.so")):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            rt = None
    if rt is None:
        pytest.skip("CUDA runtime library not found")
    pool = ctypes.c_void_p()
    dev = ctypes.c_int()
    assert rt.cudaGetDevice(ctypes.byref(dev)) == 0
    assert rt.cudaDeviceGetDefaultMemPool(ctypes.byref(pool), dev) == 0
    used_current = 7                            # cudaMemPoolAttrUsedMemCurrent
    used_high = 8                               # cudaMemPoolAttrUsedMemHigh

    def get(attr):
        v = ctypes.c_uint64(0)
        assert rt.cudaMemPoolGetAttribute(pool, attr, ctypes.byref(v)) == 0
        return v.value

    def reset():
        zero = ctypes.c_uint64(0)
        assert rt.cudaMemPoolSetAttribute(pool, used_high, ctypes.byref(zero)) == 0

    return (lambda: get(used_current)), reset, (lambda: get(used_high))


def test_noalloc_draws_nothing_from_the_memory_pool(lib):
    import torch
    shape = (1, 4096, 32, 128)
    x = torch.from_numpy(_bf16(shape, 3, True).view(np.int16)).view(torch.bfloat16).cuda()
    signs = torch.from_numpy(S.rotation_signs(128)).cuda()
    out = torch.empty(shape, dtype=torch.uint8, device="cuda")
    d = torch.empty(1, device="cuda")
    current, reset, high = _default_pool_used_high()
    torch.cuda.synchronize()
    in_use = current()                          # whatever other code holds in the pool
    reset()                                     # high water mark := memory in use
    assert lib.zyfa_quantize_noalloc(x, signs, 1, 0.0, out, d, None, *shape) == lib.ZYFA_OK
    torch.cuda.synchronize()
    assert high() == in_use
    assert lib.zyfa_quantize(x, signs, 1, 0.0, out, d, None, *shape) == lib.ZYFA_OK
    torch.cuda.synchronize()
    assert high() > in_use                      # the probe sees zyfa_quantize's scratch
