"""Pins of the oracle's forward pass (CPU only).

* equality with the independent brute force of tests/brute_force.py on tiny
  inputs, every mode;
* hand-computed closed forms (two keys; a block far below the maximum);
* invariants the paper states: causality, row 0 = V[0], uniform scores give
  the prefix mean, weights sum to one, per-row score shifts cancel, and with
  unrounded probabilities the method equals fp64 softmax attention whatever
  the maximum, the threshold or the block scaling (Sec. II-B fn. 3-4,
  Sec. IV-A fn. 9, Sec. IV-B3 fn. 12, Sec. V-E fn. 18);
* fp64 attention equal to a plain numpy softmax.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
import synthetic as S
from tests import brute_force as bf


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def _tiny(B, N, Hq, Hkv, dqk, dv, seed, dtype="e4m3"):
    q = S.normal((B, N, Hq, dqk), seed, 0)
    k = S.normal((B, N, Hkv, dqk), seed, 1)
    v = S.normal((B, N, Hkv, dv), seed, 2)
    if dtype == "e4m3":
        q8, dq = S.quantize_e4m3(q)
        k8, dk = S.quantize_e4m3(k)
        v8, dvs = S.quantize_e4m3(v)
        return q8, k8, v8, (dq, dk, dvs)
    return S.to_bf16_bits(q), S.to_bf16_bits(k), S.to_bf16_bits(v), (1.0, 1.0, 1.0)


def _run(q, k, v, descale, dtype, **kw):
    B, N, Hq, dqk = q.shape
    p = oracle.make_params(dtype=dtype, B=B, Hq=Hq, Hkv=k.shape[2], N=N, d_qk=dqk,
                           d_v=v.shape[3], descale=descale, **kw)
    out, outb, lse = oracle.fwd(p, q, k, v)
    return p, out.reshape(B, Hq, N, -1).transpose(0, 2, 1, 3), outb, lse


def _brute(q, k, v, descale, p, dtype):
    return bf.forward(q, k, v, dtype=dtype, descale=descale, p_mode=p.p_mode,
                      block_scale=p.block_scale, max_mode=p.max_mode, tau=p.tau,
                      kv_block=p.kv_block, scale_block=p.scale_block,
                      denom_mode=p.denom_mode, sigma=p.sigma, beta=p.beta,
                      softmax_scale=p.softmax_scale)


@pytest.mark.parametrize("p_mode,block_scale,max_mode",
                         list(itertools.product([0, 1, 2], [0, 1], [0, 1])))
def test_fp8_matches_brute_force(p_mode, block_scale, max_mode):
    # 2 query heads sharing 1 KV head, 150 keys: two 64-key scale blocks and
    # a ragged third; kv_block 48 so the running maximum moves several times
    q, k, v, ds = _tiny(1, 150, 2, 1, 16, 8, seed=11)
    p, out, _, _ = _run(q, k, v, ds, "e4m3", p_mode=p_mode, block_scale=block_scale,
                        max_mode=max_mode, kv_block=48, scale_block=64, tau=0.125)
    ref = _brute(q, k, v, ds, p, "e4m3")
    assert _rel(out, ref) < 1e-12


@pytest.mark.parametrize("denom_mode", [0, 1])
def test_fp8_denominators_match_brute_force(denom_mode):
    q, k, v, ds = _tiny(2, 70, 2, 2, 8, 8, seed=12)
    p, out, _, _ = _run(q, k, v, ds, "e4m3", p_mode=1, denom_mode=denom_mode,
                        kv_block=32, scale_block=16, tau=0.0)
    assert _rel(out, _brute(q, k, v, ds, p, "e4m3")) < 1e-12


@pytest.mark.parametrize("max_mode", [0, 1])
def test_bf16_matches_brute_force(max_mode):
    q, k, v, ds = _tiny(1, 90, 4, 2, 8, 8, seed=13, dtype="bf16")
    p, out, _, _ = _run(q, k, v, ds, "bf16", max_mode=max_mode, kv_block=32, tau=0.5)
    assert _rel(out, _brute(q, k, v, ds, p, "bf16")) < 1e-12


def test_fp64_reference_matches_numpy_softmax():
    q, k, v, ds = _tiny(2, 40, 4, 2, 16, 8, seed=14)
    p = oracle.make_params(dtype="e4m3", B=2, Hq=4, Hkv=2, N=40, d_qk=16, d_v=8, descale=ds)
    out, _ = oracle.attn_fp64(p, q, k, v)
    out = out.reshape(2, 4, 40, 8).transpose(0, 2, 1, 3)
    ref = bf.attention_fp64(q, k, v, dtype="e4m3", descale=ds, softmax_scale=p.softmax_scale)
    assert _rel(out, ref) < 1e-13


def _codes(vals):
    return np.array([oracle.e4m3_encode(x) for x in vals], dtype=np.uint8)


def test_closed_form_two_keys():
    """Row 1 with base-2 scores (2, 1): p = 2^6, 2^5 -> O = (2 v0 + v1) / 3;
    scores (2, 1.5): lean codes 104, 100 (64, 48), exact 104, 99 (64, 44)."""
    ln2 = math.log(2.0)
    q = _codes([1.0, 1.0]).reshape(1, 2, 1, 1)
    v = _codes([1.0, 4.0]).reshape(1, 2, 1, 1)
    for k_vals, want_lean, want_exact in (([2.0, 1.0], (64, 32), (64, 32)),
                                          ([2.0, 1.5], (64, 48), (64, 44))):
        k = _codes(k_vals).reshape(1, 2, 1, 1)
        for p_mode, want in ((1, want_lean), (0, want_exact)):
            p = oracle.make_params(dtype="e4m3", B=1, Hq=1, Hkv=1, N=2, d_qk=1, d_v=1,
                                   softmax_scale=ln2, p_mode=p_mode, max_mode=0)
            out, _, lse = oracle.fwd(p, q, k, v)
            w0, w1 = want
            assert out[1, 0] == pytest.approx((w0 * 1.0 + w1 * 4.0) / (w0 + w1), rel=1e-15)
            assert out[0, 0] == 1.0
            # LSE of the rounded weights: ln(w0 + w1) + (m - sigma) ln 2
            assert lse[1] == pytest.approx(math.log(w0 + w1) + (2.0 - 6.0) * ln2, rel=1e-14)


def test_closed_form_block_scale():
    """65 keys, d_qk = 2, q = (1, 1): key 0 scores 0, keys 1..63 score -40
    (they vanish), key 64 scores -12.5 and sits alone in the second 64-key
    block.  Without scaling Lean P gives y = 8(0.5) - 0.35 -> code 4
    (4 * 2^-9); with o = 12 it gives code 100 = 48, weighted 48 * 2^-12
    (Sec. IV-B2, Fig. 5)."""
    ln2 = math.log(2.0)
    N = 65
    q = np.zeros((1, N, 1, 2), np.uint8)
    q[0, N - 1, 0, :] = oracle.e4m3_encode(1.0)
    k = np.zeros((1, N, 1, 2), np.uint8)
    k[0, 1:64, 0, 0] = oracle.e4m3_encode(-40.0)
    k[0, 64, 0, :] = _codes([-12.0, -0.5])
    v = np.zeros((1, N, 1, 1), np.uint8)
    v[0, 0, 0, 0] = oracle.e4m3_encode(1.0)
    v[0, 64, 0, 0] = oracle.e4m3_encode(2.0)
    for bs, w_last in ((0, 4 * 2.0 ** -9), (1, 48.0 * 2.0 ** -12)):
        p = oracle.make_params(dtype="e4m3", B=1, Hq=1, Hkv=1, N=N, d_qk=2, d_v=1,
                               softmax_scale=ln2, p_mode=1, block_scale=bs, max_mode=0)
        out, _, _ = oracle.fwd(p, q, k, v, rows=np.array([N - 1]))
        want = (64.0 * 1.0 + w_last * 2.0) / (64.0 + w_last)
        assert out[0, 0] == pytest.approx(want, rel=1e-15)


@pytest.mark.parametrize("p_mode", [0, 1])
def test_causality(p_mode):
    q, k, v, ds = _tiny(1, 200, 2, 2, 16, 16, seed=15)
    rows = np.array([0, 5, 63, 64, 127, 128, 199, 200, 263, 399])
    p = oracle.make_params(dtype="e4m3", B=1, Hq=2, Hkv=2, N=200, d_qk=16, d_v=16,
                           descale=ds, p_mode=p_mode)
    base, _, _ = oracle.fwd(p, q, k, v, rows)
    k2, v2 = k.copy(), v.copy()
    rng = np.random.default_rng(0)
    for r in rows:
        i = r % 200
        k2[0, i + 1:] = rng.integers(0, 126, k2[0, i + 1:].shape, dtype=np.uint8)
        v2[0, i + 1:] = rng.integers(0, 126, v2[0, i + 1:].shape, dtype=np.uint8)
        out, _, _ = oracle.fwd(p, q, k2, v2, np.array([r]))
        assert np.array_equal(out[0], base[list(rows).index(r)])
        k2[:], v2[:] = k, v


@pytest.mark.parametrize("p_mode,max_mode,dtype",
                         [(0, 0, "e4m3"), (1, 1, "e4m3"), (0, 1, "bf16")])
def test_row0_is_v0(p_mode, max_mode, dtype):
    q, k, v, ds = _tiny(2, 64, 4, 2, 16, 16, seed=16, dtype=dtype)
    B, N, Hq = 2, 64, 4
    p = oracle.make_params(dtype=dtype, B=B, Hq=Hq, Hkv=2, N=N, d_qk=16, d_v=16,
                           descale=ds, p_mode=p_mode, max_mode=max_mode)
    rows = np.array([(b * Hq + h) * N for b in range(B) for h in range(Hq)])
    out, outb, _ = oracle.fwd(p, q, k, v, rows)
    for n, r in enumerate(rows):
        b, h = divmod(r // N, Hq)
        g = h // 2
        want = ds[2] * bf.decode(v[b, 0, g], dtype)
        assert np.array_equal(out[n], want)
        assert np.array_equal(outb[n], [oracle.bf16_encode(x) for x in want])


@pytest.mark.parametrize("p_mode,block_scale", [(0, 1), (1, 1), (1, 0)])
def test_uniform_scores_give_prefix_mean(p_mode, block_scale):
    q, k, v, ds = _tiny(1, 300, 1, 1, 8, 8, seed=17)
    q = np.zeros_like(q)
    p = oracle.make_params(dtype="e4m3", B=1, Hq=1, Hkv=1, N=300, d_qk=8, d_v=8,
                           descale=ds, p_mode=p_mode, block_scale=block_scale)
    out, _, _ = oracle.fwd(p, q, k, v)
    V = bf.decode(v[0, :, 0], "e4m3") * ds[2]
    want = np.cumsum(V, axis=0) / np.arange(1, 301)[:, None]
    assert np.max(np.abs(out - want)) < 1e-13


@pytest.mark.parametrize("p_mode,max_mode", [(0, 0), (1, 1), (1, 0)])
def test_weights_sum_to_one(p_mode, max_mode):
    q, k, v, ds = _tiny(1, 300, 2, 2, 16, 4, seed=18)
    v = np.full_like(v, oracle.e4m3_encode(1.0))
    p = oracle.make_params(dtype="e4m3", B=1, Hq=2, Hkv=2, N=300, d_qk=16, d_v=4,
                           descale=(ds[0], ds[1], 1.0), p_mode=p_mode, max_mode=max_mode)
    out, _, _ = oracle.fwd(p, q, k, v)
    assert np.max(np.abs(out - 1.0)) < 1e-6


def test_unrounded_method_equals_fp64_attention():
    """With p unrounded, sigma, tau, block exponents and the running maximum
    all cancel in acc / l, leaving softmax attention."""
    q, k, v, ds = _tiny(1, 260, 2, 1, 16, 16, seed=19)
    p = oracle.make_params(dtype="e4m3", B=1, Hq=2, Hkv=1, N=260, d_qk=16, d_v=16, descale=ds)
    ref, ref_lse = oracle.attn_fp64(p, q, k, v)
    for max_mode, tau, bs, kvb in ((0, 0.0, 1, 128), (1, 0.125, 1, 128), (1, 8.0, 0, 32),
                                   (1, 0.0, 1, 64)):
        p = oracle.make_params(dtype="e4m3", B=1, Hq=2, Hkv=1, N=260, d_qk=16, d_v=16,
                               descale=ds, p_mode=2, max_mode=max_mode, tau=tau,
                               block_scale=bs, kv_block=kvb)
        out, _, lse = oracle.fwd(p, q, k, v)
        assert _rel(out, ref) < 1e-12
        assert np.max(np.abs(lse - ref_lse)) < 1e-10


def test_gqa_head_mapping():
    """Query head h reads KV head h // (Hq/Hkv): same result as MHA with the
    KV heads repeated."""
    q, k, v, ds = _tiny(1, 70, 4, 2, 16, 8, seed=20)
    p = oracle.make_params(dtype="e4m3", B=1, Hq=4, Hkv=2, N=70, d_qk=16, d_v=8, descale=ds)
    out, _, _ = oracle.fwd(p, q, k, v)
    p2 = oracle.make_params(dtype="e4m3", B=1, Hq=4, Hkv=4, N=70, d_qk=16, d_v=8, descale=ds)
    out2, _, _ = oracle.fwd(p2, q, np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2))
    assert np.array_equal(out, out2)


def test_score_shift_cancels_without_rounding():
    """Adding the same vector c to every key adds q.c to every score of a
    row; with unrounded p the output is unchanged (Sec. V-E, fn. 18).
    Inputs are small dyadic numbers so that k + c is exact in BF16."""
    rng = np.random.default_rng(3)
    qf = (rng.integers(-8, 8, (1, 100, 1, 4)) / 4.0).astype(np.float32)
    kf = (rng.integers(-8, 8, (1, 100, 1, 4)) / 4.0).astype(np.float32)
    vf = rng.standard_normal((1, 100, 1, 4)).astype(np.float32)
    c = np.array([0.5, -0.25, 0.125, 1.0], np.float32)
    q, k, v, k2 = (S.to_bf16_bits(x) for x in (qf, kf, vf, kf + c))
    assert np.array_equal(bf.decode(k2, "bf16"), (kf + c).astype(np.float64))
    p = oracle.make_params(dtype="bf16", B=1, Hq=1, Hkv=1, N=100, d_qk=4, d_v=4, p_mode=2)
    a, _, _ = oracle.fwd(p, q, k, v)
    b, _, _ = oracle.fwd(p, q, k2, v)
    assert _rel(a, b) < 1e-12


def test_block_scaling_keeps_far_blocks():
    """Fig. 5: blocks 11-15 binades below the row maximum.  Unscaled and
    without the shift (sigma = 0) exact P rounds every such block to zero;
    with block scaling each block's maximum maps to 2^sigma and the block
    keeps its exact weight 2^-gap."""
    ln2 = math.log(2.0)
    gaps = [11.0, 12.0, 13.0, 14.0, 15.0]
    N = 64 * (1 + len(gaps))
    kv = np.zeros(N)
    for n, gap in enumerate(gaps):
        kv[64 * (n + 1):64 * (n + 2)] = -gap
    k = _codes(kv).reshape(1, N, 1, 1)
    q = np.zeros((1, N, 1, 1), np.uint8)
    q[0, N - 1, 0, 0] = oracle.e4m3_encode(1.0)
    total = 1.0 + sum(2.0 ** -g for g in gaps)
    for n in range(len(gaps) + 1):
        v = np.zeros((1, N, 1, 1), np.uint8)
        v[0, 64 * n:64 * (n + 1)] = oracle.e4m3_encode(1.0)
        row = np.array([N - 1])
        p = oracle.make_params(dtype="e4m3", B=1, Hq=1, Hkv=1, N=N, d_qk=1, d_v=1,
                               softmax_scale=ln2, p_mode=0, block_scale=0, max_mode=0,
                               sigma=0.0)
        unscaled = oracle.fwd(p, q, k, v, rows=row)[0][0, 0]
        assert unscaled == (1.0 if n == 0 else 0.0)
        for sigma in (0.0, 6.0):
            p = oracle.make_params(dtype="e4m3", B=1, Hq=1, Hkv=1, N=N, d_qk=1, d_v=1,
                                   softmax_scale=ln2, p_mode=0, block_scale=1, max_mode=0,
                                   sigma=sigma)
            scaled = oracle.fwd(p, q, k, v, rows=row)[0][0, 0]
            want = (1.0 if n == 0 else 2.0 ** -gaps[n - 1]) / total
            assert scaled == pytest.approx(want, rel=1e-12)


def test_lse_close_to_fp64(golden):
    """Sec. IV-B3: Lean P's LSE stays within a few hundredths of a nat of the
    fp64 LSE in the worst row of Gaussian inputs."""
    wl = S.Workload("t", 1, 2, 2, 2048, 128, 128)
    inp = S.make_inputs(wl)
    p = oracle.make_params(dtype="e4m3", B=1, Hq=2, Hkv=2, N=2048, d_qk=128, d_v=128,
                           descale=inp.descale, p_mode=1)
    rows = S.sample_rows(wl, per_head=256)
    _, _, lse = oracle.fwd(p, inp.q8, inp.k8, inp.v8, rows)
    _, ref = oracle.attn_fp64(p, inp.q8, inp.k8, inp.v8, rows)
    worst = np.max(np.abs(lse - ref))
    assert worst <= golden["lse_worst_row_nats"]["range"][1]


# ---------------------------------------------------------------------------
# 'mixed': BF16 Q and K, e4m3 V, FP8 probabilities
# ---------------------------------------------------------------------------
def _tiny_mixed(B, N, Hq, Hkv, dqk, dv, seed):
    q = S.normal((B, N, Hq, dqk), seed, 0)
    k = S.normal((B, N, Hkv, dqk), seed, 1)
    v = S.normal((B, N, Hkv, dv), seed, 2)
    v8, dvs = S.quantize_e4m3(v)
    return S.to_bf16_bits(q), S.to_bf16_bits(k), v8, (1.0, 1.0, dvs)


@pytest.mark.parametrize("p_mode,block_scale,max_mode",
                         list(itertools.product([0, 1, 2], [0, 1], [0, 1])))
def test_mixed_matches_brute_force(p_mode, block_scale, max_mode):
    q, k, v, ds = _tiny_mixed(1, 150, 2, 1, 16, 8, seed=31)
    p, out, _, _ = _run(q, k, v, ds, "mixed", p_mode=p_mode, block_scale=block_scale,
                        max_mode=max_mode, kv_block=48, scale_block=64, tau=0.125)
    assert p.dtype == 2 and p.descale_q == 1.0 and p.descale_k == 1.0
    assert _rel(out, _brute(q, k, v, ds, p, "mixed")) < 1e-12


def test_mixed_unrounded_equals_fp64_attention():
    q, k, v, ds = _tiny_mixed(1, 200, 2, 1, 16, 16, seed=32)
    p = oracle.make_params(dtype="mixed", B=1, Hq=2, Hkv=1, N=200, d_qk=16, d_v=16, descale=ds)
    ref, _ = oracle.attn_fp64(p, q, k, v)
    ref_np = bf.attention_fp64(q, k, v, dtype="mixed", descale=ds, softmax_scale=p.softmax_scale)
    assert _rel(ref.reshape(1, 2, 200, 16).transpose(0, 2, 1, 3), ref_np) < 1e-13
    p2 = oracle.make_params(dtype="mixed", B=1, Hq=2, Hkv=1, N=200, d_qk=16, d_v=16,
                            descale=ds, p_mode=2)
    out, _, _ = oracle.fwd(p2, q, k, v)
    assert _rel(out, ref) < 1e-12


@pytest.mark.parametrize("p_mode", [0, 1])
def test_mixed_equals_e4m3_on_shared_values(p_mode):
    """Q and K values that e4m3 and BF16 both hold exactly (e4m3 codes decoded
    into BF16): the mixed path must equal the e4m3 path with unit Q/K
    descales, since only the loads differ."""
    q8, k8, v8, (_, _, dvs) = _tiny(1, 140, 2, 2, 16, 8, seed=33)
    tab = oracle.e4m3_decode_table()
    q16 = S.to_bf16_bits(tab[q8].astype(np.float32))
    k16 = S.to_bf16_bits(tab[k8].astype(np.float32))
    _, out8, _, _ = _run(q8, k8, v8, (1.0, 1.0, dvs), "e4m3", p_mode=p_mode)
    _, outm, _, _ = _run(q16, k16, v8, (1.0, 1.0, dvs), "mixed", p_mode=p_mode)
    assert np.array_equal(out8, outm)


# ---------------------------------------------------------------------------
# key ranges and the merge of partial results (Sec. IV-B3)
# ---------------------------------------------------------------------------
def _run_range(q, k, v, ds, dtype, kb, ke, **kw):
    B, N, Hq, dqk = q.shape
    p = oracle.make_params(dtype=dtype, B=B, Hq=Hq, Hkv=k.shape[2], N=N, d_qk=dqk,
                           d_v=v.shape[3], descale=ds, key_begin=kb, key_end=ke, **kw)
    out, outb, lse = oracle.fwd(p, q, k, v)
    return p, out, lse


def test_full_key_range_equals_forward():
    q, k, v, ds = _tiny(1, 200, 2, 1, 16, 8, seed=41)
    _, out_full, lse_full = _run_range(q, k, v, ds, "e4m3", 0, 200)
    p = oracle.make_params(dtype="e4m3", B=1, Hq=2, Hkv=1, N=200, d_qk=16, d_v=8, descale=ds)
    out, _, lse = oracle.fwd(p, q, k, v)
    assert np.array_equal(out_full, out) and np.array_equal(lse_full, lse)


@pytest.mark.parametrize("p_mode,block_scale", [(0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("kb,ke", [(0, 128), (128, 256), (128, 300), (256, 300)])
def test_key_range_matches_brute_force(p_mode, block_scale, kb, ke):
    q, k, v, ds = _tiny(1, 300, 2, 1, 16, 8, seed=42)
    p, out, _ = _run_range(q, k, v, ds, "e4m3", kb, ke, p_mode=p_mode, block_scale=block_scale,
                           kv_block=128, scale_block=64)
    ref = bf.forward(q, k, v, dtype="e4m3", descale=ds, p_mode=p.p_mode,
                     block_scale=p.block_scale, max_mode=p.max_mode, tau=p.tau,
                     kv_block=p.kv_block, scale_block=p.scale_block, denom_mode=p.denom_mode,
                     sigma=p.sigma, beta=p.beta, softmax_scale=p.softmax_scale,
                     key_begin=kb, key_end=ke)
    out = out.reshape(1, 2, 300, 8).transpose(0, 2, 1, 3)
    assert _rel(out, ref) < 1e-12
    # rows that see no key of the range: zero output
    if kb > 0:
        assert not out[:, :kb].any()


def test_empty_range_gives_zero_and_minus_inf():
    q, k, v, ds = _tiny(1, 256, 1, 1, 16, 8, seed=43)
    _, out, lse = _run_range(q, k, v, ds, "e4m3", 128, 256)
    out = out.reshape(256, 8)
    assert not out[:128].any() and np.all(np.isneginf(lse[:128]))
    assert np.all(np.isfinite(lse[128:]))


@pytest.mark.parametrize("dtype", ["e4m3", "bf16"])
def test_merge_of_unrounded_ranges_is_fp64_attention(dtype):
    """With unrounded p each range is exact softmax attention over its keys,
    and the LSE-weighted merge of softmax over disjoint key sets is softmax
    over their union: the merge must give fp64 attention and its LSE."""
    q, k, v, ds = _tiny(2, 320, 2, 1, 16, 8, seed=44, dtype=dtype)
    p = oracle.make_params(dtype=dtype, B=2, Hq=2, Hkv=1, N=320, d_qk=16, d_v=8, descale=ds)
    ref, ref_lse = oracle.attn_fp64(p, q, k, v)
    parts = [_run_range(q, k, v, ds, dtype, kb, ke, p_mode=2)[1:]
             for kb, ke in ((0, 128), (128, 256), (256, 320))]
    out, lse = oracle.merge([o for o, _ in parts], [l for _, l in parts])
    assert _rel(out, ref) < 1e-12
    assert np.max(np.abs(lse - ref_lse)) < 1e-10
    # and the fp64 reference over ranges merges to the same
    ref_parts = []
    for kb, ke in ((0, 128), (128, 256), (256, 320)):
        pr = oracle.make_params(dtype=dtype, B=2, Hq=2, Hkv=1, N=320, d_qk=16, d_v=8,
                                descale=ds, key_begin=kb, key_end=ke)
        ref_parts.append(oracle.attn_fp64(pr, q, k, v))
    out2, lse2 = oracle.merge([o for o, _ in ref_parts], [l for _, l in ref_parts])
    assert _rel(out2, ref) < 1e-12 and np.max(np.abs(lse2 - ref_lse)) < 1e-10


def test_merge_single_part_is_identity():
    rng = np.random.default_rng(3)
    o = rng.standard_normal((10, 4))
    l = rng.standard_normal(10)
    l[3] = -np.inf
    out, L = oracle.merge([o], [l])
    assert np.allclose(out[np.isfinite(l)], o[np.isfinite(l)], rtol=0, atol=1e-15)
    assert np.array_equal(L, l) and not out[3].any()
