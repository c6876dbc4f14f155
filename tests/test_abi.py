"""The C ABI library builds, loads and exports every symbol include/zyfa.h
declares; argument errors are reported before anything is launched.  No
compute call is made here, so these run without a GPU."""
import os
import re

import pytest

import fp8_causal_flashattention_gb300 as Z

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    Z.build()
    return Z.load()


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(zyfa_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"zyfa_fwd", "zyfa_fwd_bf16", "zyfa_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(Z.EXPORTS) <= set(names)


def test_status_strings(lib):
    for s in range(0, -7, -1):
        assert Z.zyfa_status_string(s) != "unknown status"
    assert Z.zyfa_status_string(-99) == "unknown status"
    assert Z.zyfa_version() >= 100


FAKE = 1 << 20          # 16-byte aligned, never dereferenced: checks fail first


@pytest.mark.parametrize("args,want", [
    (dict(N=100), Z.ZYFA_ERR_SHAPE),               # N % 128
    (dict(Hq=3, Hkv=2), Z.ZYFA_ERR_SHAPE),         # Hq % Hkv
    (dict(B=-1), Z.ZYFA_ERR_SHAPE),
    (dict(Hq=0), Z.ZYFA_ERR_SHAPE),
    (dict(causal=2), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(causal=-1), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(d_qk=64), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(d_v=192), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(p_mode=2), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(block_scale=3), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(q=0), Z.ZYFA_ERR_NULL),
    (dict(out=0), Z.ZYFA_ERR_NULL),
    (dict(k=FAKE + 8), Z.ZYFA_ERR_ALIGN),
    (dict(dq=FAKE + 2), Z.ZYFA_ERR_ALIGN),
    (dict(N=1 << 30, Hq=1 << 11, Hkv=1), Z.ZYFA_ERR_SHAPE),   # byte stride >= 2^40
])
def test_fp8_argument_errors(lib, args, want):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dq=None, dk=None, dv=None, out=FAKE, B=1, Hq=2, Hkv=1,
             N=256, d_qk=128, d_v=128, causal=1, p_mode=1, block_scale=1)
    a.update(args)
    rc = lib.zyfa_fwd(a["q"], a["k"], a["v"], a["dq"], a["dk"], a["dv"], a["out"], a["B"],
                      a["Hq"], a["Hkv"], a["N"], a["d_qk"], a["d_v"], a["causal"],
                      a["p_mode"], a["block_scale"], None)
    assert rc == want


@pytest.mark.parametrize("args,want", [
    (dict(N=64), Z.ZYFA_ERR_SHAPE),
    (dict(causal=2), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(v=0), Z.ZYFA_ERR_NULL),
    (dict(out=FAKE + 4), Z.ZYFA_ERR_ALIGN),
])
def test_bf16_argument_errors(lib, args, want):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, B=2, Hq=4, Hkv=4, N=512, d_qk=192, d_v=128,
             causal=1)
    a.update(args)
    rc = lib.zyfa_fwd_bf16(a["q"], a["k"], a["v"], a["out"], a["B"], a["Hq"], a["Hkv"],
                           a["N"], a["d_qk"], a["d_v"], a["causal"], None)
    assert rc == want


@pytest.mark.parametrize("B,N", [(0, 256), (2, 0)])
def test_empty_problem_is_ok_without_launch(lib, B, N):
    assert lib.zyfa_fwd(None, None, None, None, None, None, None, B, 4, 4, N, 128, 128,
                        1, 1, 1, None) == Z.ZYFA_OK
    assert lib.zyfa_fwd_bf16(None, None, None, None, B, 4, 4, N, 128, 128, 1, None) == Z.ZYFA_OK


@pytest.mark.parametrize("args,want", [
    (dict(D=64), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(D=256), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(smooth=2), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(static=3.0), Z.ZYFA_ERR_UNSUPPORTED),          # not a power of two
    (dict(static=-2.0), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(static=2.0 ** -127), Z.ZYFA_ERR_UNSUPPORTED),  # below the FP32-normal floor
    (dict(static=float("inf")), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(B=-1), Z.ZYFA_ERR_SHAPE),
    (dict(H=-3), Z.ZYFA_ERR_SHAPE),
    (dict(descale_out=0), Z.ZYFA_ERR_NULL),
    (dict(x=0), Z.ZYFA_ERR_NULL),
    (dict(out=0), Z.ZYFA_ERR_NULL),
    (dict(x=FAKE + 8), Z.ZYFA_ERR_ALIGN),
    (dict(out=FAKE + 4), Z.ZYFA_ERR_ALIGN),
    (dict(signs=FAKE + 2), Z.ZYFA_ERR_ALIGN),
    (dict(mean=FAKE + 4), Z.ZYFA_ERR_ALIGN),
    (dict(descale_out=FAKE + 1), Z.ZYFA_ERR_ALIGN),
])
def test_quantize_argument_errors(lib, args, want):
    a = dict(x=FAKE, signs=FAKE, smooth=1, static=0.0, out=FAKE, descale_out=FAKE, mean=None,
             B=1, N=100, H=2, D=128)
    a.update(args)
    rc = Z.zyfa_quantize(a["x"], a["signs"], a["smooth"], a["static"], a["out"],
                         a["descale_out"], a["mean"], a["B"], a["N"], a["H"], a["D"], 0)
    assert rc == want


def test_quantize_noalloc_rejects_oversize_before_launch(lib):
    """zyfa_quantize_noalloc: a smoothing call whose partial sums exceed the
    library's 16 MiB buffer returns ZYFA_ERR_SCRATCH before anything is
    launched (the pointers are never dereferenced, no GPU is needed)."""
    B, N, H, D = 4096, 4, 128, 192            # 4 x 4096 x 128 x 192 bytes of partial sums
    rc = Z.zyfa_quantize_noalloc(FAKE, None, 1, 0.0, FAKE, FAKE, FAKE, B, N, H, D, 0)
    assert rc == Z.ZYFA_ERR_SCRATCH
    assert "scratch" in Z.zyfa_status_string(rc)
    # without smoothing and with a static scale no scratch is needed: the
    # NULL x is reported first
    assert Z.zyfa_quantize_noalloc(None, None, 0, 1.0, FAKE, FAKE, None, B, N, H, D, 0) == Z.ZYFA_ERR_NULL


def _bshd(B, N, H, d):
    return [N * H * d, H * d, d]


@pytest.mark.parametrize("which,bad,want", [
    ("q", [4096 * 2 * 128, 2 * 128, 120], Z.ZYFA_ERR_ALIGN),     # head stride 120 B
    ("k", [-1, 128, 128], Z.ZYFA_ERR_SHAPE),
    ("v", [0, 128, 128], Z.ZYFA_ERR_SHAPE),
    ("o", [256 * 2 * 128, 2 * 128, 124], Z.ZYFA_ERR_ALIGN),     # 248 B: not 16-byte aligned
    ("q", [1 << 40, 256, 128], Z.ZYFA_ERR_SHAPE),                # byte stride >= 2^40
    ("o", [1 << 39, 256, 128], Z.ZYFA_ERR_SHAPE),                # 2^40 bytes: the output's tensor map
])
def test_strided_argument_errors(lib, which, bad, want):
    st = {"q": _bshd(1, 256, 2, 128), "k": _bshd(1, 256, 1, 128), "v": _bshd(1, 256, 1, 128),
          "o": [256 * 2 * 128, 2 * 128, 128]}
    st[which] = bad
    flat = st["q"] + st["k"] + st["v"] + st["o"]
    rc = Z.zyfa_fwd_strided(FAKE, FAKE, FAKE, None, None, None, FAKE, None, 1, 2, 1, 256, 128, 128,
                            1, 1, 1, flat, 0)
    assert rc == want


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("kb,ke,lse,want", [
    (64, 256, FAKE, Z.ZYFA_ERR_SHAPE),       # not a multiple of 128
    (0, 200, FAKE, Z.ZYFA_ERR_SHAPE),
    (256, 128, FAKE, Z.ZYFA_ERR_SHAPE),      # end before begin
    (-128, 128, FAKE, Z.ZYFA_ERR_SHAPE),
    (0, 512, FAKE, Z.ZYFA_ERR_SHAPE),        # past N
    (0, 256, 0, Z.ZYFA_ERR_NULL),            # the LSE is required
])
def test_partial_argument_errors(lib, fp8, kb, ke, lse, want):
    N = 256
    if fp8:
        rc = Z.zyfa_fwd_partial(FAKE, FAKE, FAKE, None, None, None, FAKE, lse, 1, 2, 1, N, 128,
                                128, key_begin=kb, key_end=ke, stream=0)
    else:
        rc = Z.zyfa_fwd_bf16_partial(FAKE, FAKE, FAKE, FAKE, lse, 1, 2, 1, N, 128, 128,
                                     key_begin=kb, key_end=ke, stream=0)
    assert rc == want


def test_partial_empty_problem_is_ok(lib):
    assert Z.zyfa_fwd_partial(0, 0, 0, None, None, None, 0, None, 0, 2, 1, 256, 128, 128,
                              key_begin=0, key_end=256, stream=0) == Z.ZYFA_OK
    assert Z.zyfa_fwd_bf16_partial(0, 0, 0, 0, None, 1, 2, 1, 0, 128, 128, key_begin=0,
                                   key_end=0, stream=0) == Z.ZYFA_OK


@pytest.mark.parametrize("kw,want", [
    (dict(outs=[], lses=[]), Z.ZYFA_ERR_SHAPE),
    (dict(outs=[FAKE] * 17, lses=[FAKE] * 17), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(outs=[FAKE, 0], lses=[FAKE, FAKE]), Z.ZYFA_ERR_NULL),
    (dict(outs=[FAKE, FAKE], lses=[FAKE, 0]), Z.ZYFA_ERR_NULL),
    (dict(out=0), Z.ZYFA_ERR_NULL),
    (dict(outs=[FAKE, FAKE + 8], lses=[FAKE, FAKE]), Z.ZYFA_ERR_ALIGN),
    (dict(lses=[FAKE, FAKE + 2]), Z.ZYFA_ERR_ALIGN),
    (dict(out=FAKE + 4), Z.ZYFA_ERR_ALIGN),
    (dict(lse=FAKE + 1), Z.ZYFA_ERR_ALIGN),
    (dict(d_v=12), Z.ZYFA_ERR_SHAPE),
    (dict(d_v=24), Z.ZYFA_ERR_SHAPE),                    # not a power of two
    (dict(N=1 << 30, Hq=2), Z.ZYFA_ERR_SHAPE),           # B Hq N >= 2^31
    (dict(d_v=0), Z.ZYFA_ERR_SHAPE),
    (dict(Hq=0), Z.ZYFA_ERR_SHAPE),
    (dict(B=-1), Z.ZYFA_ERR_SHAPE),
])
def test_merge_argument_errors(lib, kw, want):
    a = dict(outs=[FAKE, FAKE], lses=[FAKE, FAKE + 4096], out=FAKE, lse=None, B=1, Hq=2, N=256,
             d_v=128)
    a.update(kw)
    assert Z.zyfa_merge(a["outs"], a["lses"], a["out"], a["lse"], a["B"], a["Hq"], a["N"],
                        a["d_v"], stream=0) == want


def test_merge_empty_problem_is_ok(lib):
    assert Z.zyfa_merge([FAKE], [FAKE], FAKE, None, 0, 2, 256, 128, stream=0) == Z.ZYFA_OK
    assert Z.zyfa_merge([FAKE], [FAKE], FAKE, None, 1, 2, 0, 128, stream=0) == Z.ZYFA_OK


def _r256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("B,Hq,Hkv,N,dqk,dv,lse", [
    (1, 32, 32, 32768, 128, 128, 0), (2, 8, 2, 384, 192, 128, 1), (3, 6, 3, 128, 128, 128, 1),
    (0, 4, 4, 256, 128, 128, 1), (1, 1, 1, 0, 128, 128, 0)])
def test_host_workspace_bytes(lib, B, Hq, Hkv, N, dqk, dv, lse):
    bn = B * N
    want = (_r256(bn * Hq * dqk) + _r256(bn * Hkv * dqk) + _r256(bn * Hkv * dv) +
            _r256(bn * Hq * dv * 2) + (_r256(bn * Hq * 4) if lse else 0) + 256)
    assert Z.zyfa_fwd_host_workspace_bytes(B, Hq, Hkv, N, dqk, dv, lse) == want


@pytest.mark.parametrize("bad", [dict(B=-1), dict(Hq=0), dict(Hkv=0), dict(N=-128)])
def test_host_workspace_bytes_rejects(lib, bad):
    a = dict(B=1, Hq=4, Hkv=4, N=256, d_qk=128, d_v=128)
    a.update(bad)
    assert Z.zyfa_fwd_host_workspace_bytes(a["B"], a["Hq"], a["Hkv"], a["N"], a["d_qk"],
                                           a["d_v"], 0) == 0


HOST = 0x10000                                 # never dereferenced: every case fails first


@pytest.mark.parametrize("kw,want", [
    (dict(B=-1), Z.ZYFA_ERR_SHAPE),
    (dict(Hkv=3), Z.ZYFA_ERR_SHAPE),                     # Hq % Hkv
    (dict(N=200), Z.ZYFA_ERR_SHAPE),
    (dict(causal=2), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(d_qk=64), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(p_mode=7), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(block_scale=2), Z.ZYFA_ERR_UNSUPPORTED),
    (dict(n_chunks=-1), Z.ZYFA_ERR_SHAPE),
    (dict(n_chunks=33), Z.ZYFA_ERR_SHAPE),
    (dict(q=None), Z.ZYFA_ERR_NULL),
    (dict(out=None), Z.ZYFA_ERR_NULL),
    (dict(workspace=None), Z.ZYFA_ERR_NULL),
    (dict(workspace=FAKE + 16), Z.ZYFA_ERR_ALIGN),       # 256-byte alignment
    (dict(workspace_bytes=-1), Z.ZYFA_ERR_SCRATCH),      # one byte short
    (dict(lse=HOST, workspace_bytes=0), Z.ZYFA_ERR_SCRATCH),   # the LSE needs room too
    (dict(B=1 << 20, N=1 << 16, Hq=8, Hkv=8), Z.ZYFA_ERR_SHAPE),   # B Hq N/128 >= 2^31
])
def test_host_argument_errors(lib, kw, want):
    a = dict(q=HOST, k=HOST, v=HOST, descale=None, out=HOST, lse=None, B=1, Hq=4, Hkv=2, N=256,
             d_qk=128, d_v=128, causal=1, p_mode=Z.ZYFA_P_LEAN, block_scale=1, n_chunks=0,
             workspace=FAKE, workspace_bytes=0)
    a.update(kw)
    if a["workspace_bytes"] <= 0:                # relative to what the shape needs
        a["workspace_bytes"] += Z.zyfa_fwd_host_workspace_bytes(
            a["B"], a["Hq"], a["Hkv"], a["N"], a["d_qk"], a["d_v"], 0)
    assert Z.zyfa_fwd_host(a["q"], a["k"], a["v"], a["descale"], a["out"], a["lse"], a["B"],
                           a["Hq"], a["Hkv"], a["N"], a["d_qk"], a["d_v"], a["causal"],
                           a["p_mode"], a["block_scale"], a["n_chunks"], a["workspace"],
                           a["workspace_bytes"], stream=0) == want


def test_host_empty_problem_is_ok(lib):
    for B, N in ((0, 256), (1, 0)):
        assert Z.zyfa_fwd_host(None, None, None, None, None, None, B, 4, 2, N, 128, 128, 1,
                               Z.ZYFA_P_LEAN, 1, 0, None, 0, stream=0) == Z.ZYFA_OK


def _check_plan(B, Hq, Hkv, n):
    G = Hq // Hkv
    plan = Z.zyfa_fwd_host_plan(B, Hq, Hkv, n)
    assert isinstance(plan, list) and 1 <= len(plan) <= max(2 * (n or 16) - 1, 1)
    seen = {}
    copied = set()
    for c, (b0, nb, g0, hk, h0, hq, kv) in enumerate(plan):
        assert nb >= 1 and hk >= 1 and hq >= 1 and hq % hk == 0
        assert 0 <= b0 and b0 + nb <= B and 0 <= g0 and g0 + hk <= Hkv
        assert 0 <= h0 and h0 + hq <= Hq
        r = hq // hk
        for hl in range(hq):
            # the kernel's view maps local query head hl to local K/V head
            # hl // (hq / hk): it must be the global head's own K/V head
            assert (h0 + hl) // G == g0 + hl // r
        for b in range(b0, b0 + nb):
            for g in range(g0, g0 + hk):
                if kv:
                    assert (b, g) not in copied
                    copied.add((b, g))
                else:
                    assert (b, g) in copied              # copied by an earlier chunk
            for h in range(h0, h0 + hq):
                assert (b, h) not in seen
                seen[(b, h)] = c
    assert len(seen) == B * Hq and len(copied) == B * Hkv


@pytest.mark.parametrize("B,Hq,Hkv", [
    (1, 32, 32), (1, 32, 8), (1, 32, 1), (2, 32, 8), (3, 8, 2), (1, 128, 128), (1, 7, 7),
    (1, 64, 2), (4, 32, 32), (5, 12, 3), (17, 4, 4), (1, 1, 1), (2, 6, 1), (1, 96, 3)])
@pytest.mark.parametrize("n", [0, 1, 2, 3, 4, 7, 8, 16, 31, 32])
def test_host_plan_partitions_the_problem(lib, B, Hq, Hkv, n):
    _check_plan(B, Hq, Hkv, n)


def test_host_plan_shapes_used_by_the_bench(lib):
    # B=1, 32 heads, 16 chunks of 2 heads; one K/V head: query sub-ranges
    assert [c[5] for c in Z.zyfa_fwd_host_plan(1, 32, 32, 16)] == [2] * 16
    p = Z.zyfa_fwd_host_plan(1, 32, 1, 16)
    assert [c[4] for c in p] == list(range(0, 32, 2)) and [c[6] for c in p] == [1] + [0] * 15


@pytest.mark.parametrize("args,want", [
    ((0, 4, 4, 0), Z.ZYFA_ERR_SHAPE), ((1, 0, 1, 0), Z.ZYFA_ERR_SHAPE),
    ((1, 6, 4, 0), Z.ZYFA_ERR_SHAPE), ((1, 4, 4, -1), Z.ZYFA_ERR_SHAPE),
    ((1, 4, 4, 33), Z.ZYFA_ERR_SHAPE)])
def test_host_plan_errors(lib, args, want):
    assert Z.zyfa_fwd_host_plan(*args) == want
    assert Z.load().zyfa_fwd_host_plan(1, 4, 4, 0, None, 3) == Z.ZYFA_ERR_NULL


def test_host_binding_rejects_device_or_strided_tensors(lib):
    import torch
    q = torch.zeros((1, 256, 2, 128), dtype=torch.uint8)
    with pytest.raises(ValueError):                  # a BHSD view is not contiguous
        Z.attention_fp8_host(q.transpose(1, 2).contiguous().transpose(1, 2), q, q)
    with pytest.raises(ValueError):                  # K's sequence length differs
        Z.attention_fp8_host(q, q[:, :128], q[:, :128])
