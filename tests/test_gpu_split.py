"""Attention over a key range (zyfa_fwd_partial / zyfa_fwd_bf16_partial) and
the LSE merge of partial results (zyfa_merge), against the oracle's key
range and its float64 merge (Sec. IV-B3: the LSE lets results over
different key ranges be merged)."""
import numpy as np
import pytest

import oracle
import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

MODES = ["lean", "exact", "lean_nobs", "bf16"]
CASES = [
    # name, B, Hq, Hkv, N, d_qk
    ("gqa", 2, 4, 2, 640, 128),
    ("mla", 1, 2, 2, 512, 192),
]
STRICT_REL_L2 = 1e-3       # as the all-rows parity tests


@pytest.fixture(scope="module")
def lib():
    import fp8_causal_flashattention_gb300 as Z
    Z.build()
    Z.load()
    return Z


def _inputs(case, mode, seed=11, kind="gaussian"):
    wl = S.Workload(case[0], *case[1:6], 128, kind=kind)
    inp = S.make_inputs(wl, seed=seed, fp8=mode != "bf16", bf16=mode == "bf16")
    return wl, inp, P.to_device(inp, mode != "bf16")


def _partial(Z, dev, mode, kb, ke):
    (q, k, v), ds = dev
    if mode == "bf16":
        return Z.attention_partial(q, k, v, key_begin=kb, key_end=ke)
    return Z.attention_partial(q, k, v, ds[0], ds[1], ds[2], key_begin=kb, key_end=ke,
                               p_mode=Z.ZYFA_P_LEAN if mode.startswith("lean") else Z.ZYFA_P_EXACT,
                               block_scale=0 if mode.endswith("nobs") else 1)


def _ranges(N):
    h = (N // 256) * 128
    return [(0, h), (h, N), (128, 384), (N - 128, N), (256, 256)]


def _decoded(out, lse, wl, rows):
    o = P.gather_rows(out, wl, rows)
    l = lse.reshape(-1).cpu().numpy().astype(np.float64)[rows]
    return o, l


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("mode", MODES)
def test_key_range_matches_oracle(lib, case, mode):
    wl, inp, dev = _inputs(case, mode)
    rows = np.arange(wl.B * wl.Hq * wl.N)
    q, k, v = P.qkv_for(inp, mode)
    for kb, ke in _ranges(wl.N):
        out, lse = _partial(lib, dev, mode, kb, ke)
        got, got_lse = _decoded(out, lse, wl, rows)
        p = P.oracle_params(wl, inp, mode, key_begin=kb, key_end=ke)
        _, ref_b, ref_lse = oracle.fwd(p, q, k, v, rows)
        ref = oracle.bf16_bits_to_f64(ref_b)
        empty = np.isneginf(ref_lse)
        # rows that see no key of the range: exactly 0 and -inf
        assert not got[empty].any() and np.all(np.isneginf(got_lse[empty])), (kb, ke)
        live = ~empty
        if not live.any():
            continue
        assert np.all(np.isfinite(got[live])) and np.all(np.isfinite(got_lse[live]))
        rel = np.linalg.norm(got[live] - ref[live]) / np.linalg.norm(ref[live])
        err = np.abs(got_lse[live] - ref_lse[live])
        print(case[0], mode, (kb, ke), "rel_l2", rel, "lse max", err.max())
        assert rel <= STRICT_REL_L2, (kb, ke, rel)
        # as the LSE tests: FP32 against fp64 may tip a lazy-rescale test
        assert err.max() <= 2e-2 and np.sqrt(np.mean(err ** 2)) <= 5e-4, (kb, ke)


@pytest.mark.parametrize("mode", ["lean", "exact", "bf16"])
def test_full_range_is_the_ordinary_call(lib, mode):
    """A partial call runs the kernel the ordinary call runs: the range
    [0, N) must give the ordinary call's output and LSE bit for bit."""
    import torch
    Z = lib
    wl, inp, dev = _inputs(("gqa", 2, 4, 2, 640, 128), mode, seed=12)
    out, lse = _partial(Z, dev, mode, 0, wl.N)
    (q, k, v), ds = dev
    if mode == "bf16":
        ref, ref_lse = Z.attention_bf16(q, k, v, return_lse=True)
    else:
        ref, ref_lse = Z.attention_fp8(q, k, v, ds[0], ds[1], ds[2],
                                       p_mode=Z.ZYFA_P_LEAN if mode == "lean" else Z.ZYFA_P_EXACT,
                                       return_lse=True)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(lse, ref_lse)


def _bf16(x):
    """Round float64 values to BF16 (nearest even) and back, as the kernels'
    output conversion does."""
    import torch
    return torch.from_numpy(np.asarray(x)).to(torch.bfloat16).to(torch.float64).numpy()


def _merge_ref(parts, wl, rows):
    outs, lses = zip(*[_decoded(o, l, wl, rows) for o, l in parts])
    return oracle.merge(list(outs), list(lses))


def _check_merge(got, got_lse, ref, ref_lse):
    """FP32 merge then one BF16 rounding, against the float64 merge of the
    same partial results: within half a BF16 step of the exact value (plus
    FP32's share), and the LSE to FP32 accuracy."""
    tol = 2.0 ** -8 * np.abs(ref) * (1 + 1e-4) + 1e-6 * np.max(np.abs(ref))
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], ref[bad][:5])
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isneginf(got_lse), ~fin)
    assert np.all(np.abs(got_lse[fin] - ref_lse[fin]) <= 2e-6 * np.maximum(1, np.abs(ref_lse[fin])))
    assert not got[~fin].any()


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("mode", MODES)
def test_merge_matches_oracle_merge(lib, case, mode):
    wl, inp, dev = _inputs(case, mode, seed=13)
    rows = np.arange(wl.B * wl.Hq * wl.N)
    cuts = [0, 128, 384, wl.N]
    parts = [_partial(lib, dev, mode, a, b) for a, b in zip(cuts[:-1], cuts[1:])]
    out, lse = lib.merge([o for o, _ in parts], [l for _, l in parts])
    got, got_lse = _decoded(out, lse, wl, rows)
    ref, ref_lse = _merge_ref(parts, wl, rows)
    _check_merge(got, got_lse, ref, ref_lse)
    # the merged result is attention over all keys: against fp64 it is about
    # as close as the ordinary call (each part adds one BF16 rounding)
    q, k, v = P.qkv_for(inp, mode)
    p = P.oracle_params(wl, inp, mode)
    ref64, ref64_lse = oracle.attn_fp64(p, q, k, v, rows)
    one = P.gather_rows(P.gpu_run(inp, mode, dev), wl, rows)
    e_merged = np.linalg.norm(got - ref64) / np.linalg.norm(ref64)
    e_one = np.linalg.norm(one - ref64) / np.linalg.norm(ref64)
    print(case[0], mode, "rel_l2 vs fp64: merged", e_merged, "one call", e_one,
          "lse", np.max(np.abs(got_lse - ref64_lse)))
    assert e_merged <= 1.25 * e_one + 2e-3
    assert np.max(np.abs(got_lse - ref64_lse)) <= (0.04 if mode != "bf16" else 1e-3)


def test_merge_of_oracle_parts_reproduces_oracle(lib):
    """The GPU merge of the kernel's parts against the oracle's own parts
    (BF16 outputs, as the kernel's) merged in float64 and rounded to BF16:
    the kernel path end to end."""
    mode = "lean"
    case = ("gqa", 2, 4, 2, 640, 128)
    wl, inp, dev = _inputs(case, mode, seed=14)
    rows = np.arange(wl.B * wl.Hq * wl.N)
    q, k, v = P.qkv_for(inp, mode)
    cuts = [0, 256, wl.N]
    parts, ref_parts = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        parts.append(_partial(lib, dev, mode, a, b))
        p = P.oracle_params(wl, inp, mode, key_begin=a, key_end=b)
        _, ob, l = oracle.fwd(p, q, k, v, rows)
        ref_parts.append((oracle.bf16_bits_to_f64(ob), l))
    out, lse = lib.merge([o for o, _ in parts], [l for _, l in parts])
    got, got_lse = _decoded(out, lse, wl, rows)
    ref, ref_lse = oracle.merge([o for o, _ in ref_parts], [l for _, l in ref_parts])
    ref = _bf16(ref)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    print("merged vs oracle merge of oracle parts", rel)
    assert rel <= STRICT_REL_L2


def test_merge_empty_parts_and_in_place(lib):
    import torch
    mode = "lean"
    wl, inp, dev = _inputs(("mla", 1, 2, 2, 512, 192), mode, seed=15)
    rows = np.arange(wl.B * wl.Hq * wl.N)
    # one part that rows < 256 never reach: they merge to 0 / -inf
    o1, l1 = _partial(lib, dev, mode, 256, wl.N)
    out, lse = lib.merge([o1], [l1])
    got, got_lse = _decoded(out, lse, wl, rows)
    ref, ref_lse = _merge_ref([(o1, l1)], wl, rows)
    _check_merge(got, got_lse, ref, ref_lse)
    assert np.all(np.isneginf(got_lse.reshape(wl.B * wl.Hq, wl.N)[:, :256]))
    # in place into the first part, with two more parts (one all-empty range)
    o0, l0 = _partial(lib, dev, mode, 0, 256)
    o2, l2 = _partial(lib, dev, mode, 128, 128)
    ref, ref_lse = _merge_ref([(o0, l0), (o1, l1), (o2, l2)], wl, rows)
    copy, copy_lse = lib.merge([o0, o1, o2], [l0, l1, l2])
    rc = lib.zyfa_merge([o0, o1, o2], [l0, l1, l2], o0, l0, wl.B, wl.Hq, wl.N, wl.d_v)
    assert rc == lib.ZYFA_OK
    torch.cuda.synchronize()
    assert bool((copy == o0).all()) and bool((copy_lse == l0).all())
    got, _ = _decoded(o0, l0, wl, rows)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) * (1 + 1e-4) + 1e-6)


def test_full_size_split_sampled_rows(lib):
    """d_qk = 128, N = 32K, 32 heads, Lean P: two halves and the merge, in the
    launch configuration of the split-key bench line; sampled rows against
    the oracle over the same ranges and its float64 merge."""
    mode = "lean"
    wl = S.WORKLOADS["d128"]
    inp = S.make_inputs(wl)
    dev = P.to_device(inp, True)
    half = wl.N // 2
    parts = [_partial(lib, dev, mode, 0, half), _partial(lib, dev, mode, half, wl.N)]
    out, lse = lib.merge([o for o, _ in parts], [l for _, l in parts])
    rows = S.sample_rows(wl, per_head=32)
    got, got_lse = _decoded(out, lse, wl, rows)
    q, k, v = P.qkv_for(inp, mode)
    ref_parts = []
    for a, b in ((0, half), (half, wl.N)):
        p = P.oracle_params(wl, inp, mode, key_begin=a, key_end=b)
        _, ob, l = oracle.fwd(p, q, k, v, rows)
        ref_parts.append((oracle.bf16_bits_to_f64(ob), l))
    ref, ref_lse = oracle.merge([o for o, _ in ref_parts], [l for _, l in ref_parts])
    ref = _bf16(ref)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    err = np.abs(got_lse - ref_lse)
    print("full size split: rel_l2", rel, "lse max", err.max())
    assert rel <= STRICT_REL_L2
    assert err.max() <= 2e-2 and np.sqrt(np.mean(err ** 2)) <= 5e-4


@pytest.mark.parametrize("mode", ["lean", "bf16"])
def test_merge_many_parts(lib, mode):
    """One part per 128-key block (5 parts, the templated kernels), and the
    same with empty parts added (12 parts, the general kernel): both against
    the float64 merge, and equal to each other (an empty part weighs 0)."""
    import torch
    wl, inp, dev = _inputs(("gqa", 2, 4, 2, 640, 128), mode, seed=16)
    rows = np.arange(wl.B * wl.Hq * wl.N)
    parts = [_partial(lib, dev, mode, a, a + 128) for a in range(0, wl.N, 128)]
    empty = [_partial(lib, dev, mode, 256, 256) for _ in range(7)]
    out5, lse5 = lib.merge([o for o, _ in parts], [l for _, l in parts])
    mixed = parts[:2] + empty + parts[2:]
    out12, lse12 = lib.merge([o for o, _ in mixed], [l for _, l in mixed])
    got, got_lse = _decoded(out5, lse5, wl, rows)
    ref, ref_lse = _merge_ref(parts, wl, rows)
    _check_merge(got, got_lse, ref, ref_lse)
    assert bool((out5 == out12).all()) and bool((lse5 == lse12).all())
