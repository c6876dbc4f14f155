"""FP8 on the sequence lengths where zyfa_fwd runs the two-query-tile
kernel -- at d_qk = 128 Lean P beyond 2048 keys and exact P beyond 4096, at
d_qk = 192 Lean P beyond 16384 (shorter ones and exact P at 192 run the
persistent one-tile kernel, which the other GPU tests cover at their sizes):
every row against the oracle, with the LSE, over a key range, without the
causal mask and with BHSD strides."""
import numpy as np
import pytest

import oracle
import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

STRICT_REL_L2 = 1e-3
N_LEAN = 4096                 # 32 query tiles: the two-tile kernel's range for Lean P
N_EXACT = 8192                # and for exact P


@pytest.fixture(scope="module")
def lib():
    import fp8_causal_flashattention_gb300 as Z
    Z.build()
    Z.load()
    return Z


def _setup(kind="gaussian", Hq=2, Hkv=1, seed=21, N=N_LEAN):
    wl = S.Workload(f"two_tile_{kind}", 1, Hq, Hkv, N, 128, 128, kind=kind)
    inp = S.make_inputs(wl, seed=seed)
    return wl, inp, P.to_device(inp)


def _mode_args(Z, mode):
    return dict(p_mode=Z.ZYFA_P_LEAN if mode.startswith("lean") else Z.ZYFA_P_EXACT,
                block_scale=0 if mode.endswith("nobs") else 1)


def _n_for(mode):
    return N_LEAN if mode.startswith("lean") else N_EXACT


def _lse_rows(lse):
    return lse.cpu().numpy().reshape(-1).astype(np.float64)       # [B, Hq, N] = row order


@pytest.mark.parametrize("kind", ["gaussian", "sink", "activation"])
@pytest.mark.parametrize("mode", ["lean", "lean_nobs", "exact", "exact_nobs"])
def test_all_rows_and_lse(lib, kind, mode):
    Z = lib
    # exact P at N = 8192 with one query head keeps the oracle's rows at 8192
    wl, inp, ((q, k, v), ds) = _setup(kind, Hq=2 if mode.startswith("lean") else 1, N=_n_for(mode))
    out, lse = Z.attention_fp8(q, k, v, ds[0], ds[1], ds[2], return_lse=True, **_mode_args(Z, mode))
    rows = np.arange(wl.B * wl.Hq * wl.N)
    res = P.errors(P.gather_rows(out, wl, rows), inp, mode, rows, extra=False)
    print(kind, mode, res)
    assert P.passes(res, mode) and res["rel_l2"] <= STRICT_REL_L2, res
    _, _, ref_lse = oracle.fwd(P.oracle_params(wl, inp, mode), inp.q8, inp.k8, inp.v8, rows)
    err = np.abs(_lse_rows(lse) - ref_lse)
    # as the LSE tests: FP32 against fp64 may tip a lazy-rescale test in a row
    assert err.max() <= 2e-2 and np.sqrt(np.mean(err ** 2)) <= 5e-4, (err.max(), np.sqrt(np.mean(err ** 2)))


@pytest.mark.parametrize("mode", ["lean", "exact"])
def test_odd_tile_count_all_rows(lib, mode):
    """An odd number of query tiles just above each mode's switch to this
    kernel (Lean P 17 tiles, exact P 33): the last CTA holds one tile and
    releases every K/V stage it reads alone; every row against the oracle,
    with the LSE."""
    Z = lib
    N = (2048 if mode == "lean" else 4096) + 128
    wl, inp, ((q, k, v), ds) = _setup("gaussian", Hq=2, Hkv=1, seed=27, N=N)
    out, lse = Z.attention_fp8(q, k, v, ds[0], ds[1], ds[2], return_lse=True, **_mode_args(Z, mode))
    rows = np.arange(wl.B * wl.Hq * wl.N)
    res = P.errors(P.gather_rows(out, wl, rows), inp, mode, rows, extra=False)
    print(mode, res)
    assert P.passes(res, mode) and res["rel_l2"] <= STRICT_REL_L2, res
    _, _, ref_lse = oracle.fwd(P.oracle_params(wl, inp, mode), inp.q8, inp.k8, inp.v8, rows)
    err = np.abs(_lse_rows(lse) - ref_lse)
    assert err.max() <= 2e-2 and np.sqrt(np.mean(err ** 2)) <= 5e-4


@pytest.mark.parametrize("kind", ["gaussian", "sink"])
def test_mla_lean_rows(lib, kind):
    """Lean P at d_qk = 192 beyond 16384 keys: the two-tile kernel with separate
    K and V rings, on an odd number of query tiles (129: the last CTA holds one
    tile, whose K and V blocks are released by its issuers alone); the first two
    and the last three tiles whole plus a seeded sample of the others against the
    oracle, with the LSE."""
    Z = lib
    N = 16384 + 128
    wl = S.Workload(f"two_tile_mla_{kind}", 1, 1, 1, N, 192, 128, kind=kind)
    inp = S.make_inputs(wl, seed=25)
    (q, k, v), ds = P.to_device(inp)
    out, lse = Z.attention_fp8(q, k, v, ds[0], ds[1], ds[2], return_lse=True, p_mode=Z.ZYFA_P_LEAN)
    mid = np.random.default_rng(7).choice(np.arange(256, N - 384), 1024, replace=False)
    rows = np.unique(np.concatenate([np.arange(256), mid, np.arange(N - 384, N)]))
    res = P.errors(P.gather_rows(out, wl, rows), inp, "lean", rows, extra=False)
    print(kind, res)
    assert P.passes(res, "lean") and res["rel_l2"] <= STRICT_REL_L2, res
    _, _, ref_lse = oracle.fwd(P.oracle_params(wl, inp, "lean"), inp.q8, inp.k8, inp.v8, rows)
    err = np.abs(_lse_rows(lse)[rows] - ref_lse)
    assert err.max() <= 2e-2 and np.sqrt(np.mean(err ** 2)) <= 5e-4


@pytest.mark.parametrize("mode", ["lean", "exact"])
def test_key_range(lib, mode):
    Z = lib
    N = _n_for(mode)
    wl, inp, ((q, k, v), ds) = _setup(seed=22, Hq=2 if mode == "lean" else 1, N=N)
    kb, ke = N // 4, 3 * N // 4
    out, lse = Z.attention_partial(q, k, v, ds[0], ds[1], ds[2], key_begin=kb, key_end=ke, **_mode_args(Z, mode))
    rows = np.arange(wl.B * wl.Hq * wl.N)
    got = P.gather_rows(out, wl, rows)
    got_lse = _lse_rows(lse)
    p = P.oracle_params(wl, inp, mode, key_begin=kb, key_end=ke)
    _, ref_b, ref_lse = oracle.fwd(p, inp.q8, inp.k8, inp.v8, rows)
    ref = oracle.bf16_bits_to_f64(ref_b)
    empty = np.isneginf(ref_lse)
    assert empty.any() and (~empty).any()
    assert not got[empty].any() and np.all(np.isneginf(got_lse[empty]))
    live = ~empty
    rel = np.linalg.norm(got[live] - ref[live]) / np.linalg.norm(ref[live])
    err = np.abs(got_lse[live] - ref_lse[live])
    assert rel <= STRICT_REL_L2, rel
    assert err.max() <= 2e-2 and np.sqrt(np.mean(err ** 2)) <= 5e-4


@pytest.mark.parametrize("mode", ["lean", "exact"])
def test_no_causal_mask(lib, mode):
    Z = lib
    wl, inp, ((q, k, v), ds) = _setup(Hq=1, seed=23, N=_n_for(mode))
    out = Z.attention_fp8(q, k, v, ds[0], ds[1], ds[2], causal=0, **_mode_args(Z, mode))
    # every row sees every key: check a seeded sample of rows (all of them at 4096)
    rows = np.arange(wl.N) if wl.N <= 4096 else np.sort(np.random.default_rng(5).choice(wl.N, 1024, replace=False))
    res = P.errors(P.gather_rows(out, wl, rows), inp, mode, rows, extra=False, causal=0)
    print(res)
    assert P.passes(res, mode) and res["rel_l2"] <= STRICT_REL_L2, res


@pytest.mark.parametrize("mode", ["lean", "exact"])
def test_bhsd_strides_bit_identical(lib, mode):
    import torch
    Z = lib
    wl, inp, ((q, k, v), ds) = _setup(Hq=4, Hkv=2, seed=24, N=_n_for(mode))
    ref = Z.attention_fp8(q, k, v, ds[0], ds[1], ds[2], **_mode_args(Z, mode))
    qs, ks, vs = (t.transpose(1, 2).contiguous().transpose(1, 2) for t in (q, k, v))
    out = torch.empty((wl.B, wl.Hq, wl.N, wl.d_v), dtype=torch.bfloat16, device=q.device).transpose(1, 2)
    got = Z.attention_fp8(qs, ks, vs, ds[0], ds[1], ds[2], out=out, **_mode_args(Z, mode))
    assert torch.equal(got.contiguous().view(torch.int16), ref.view(torch.int16))
