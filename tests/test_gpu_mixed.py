"""BF16 QK^T with FP8 PV (zyfa_fwd_bf16qk_fp8pv) against the oracle's 'mixed'
data type, on the GPU."""
import numpy as np
import pytest

import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

STRICT_REL_L2 = 1e-3


@pytest.fixture(scope="module")
def lib():
    import fp8_causal_flashattention_gb300 as Z
    Z.build()
    Z.load()
    return Z


def _dev(inp):
    import torch
    q = torch.from_numpy(inp.q16.view(np.int16)).view(torch.bfloat16).cuda()
    k = torch.from_numpy(inp.k16.view(np.int16)).view(torch.bfloat16).cuda()
    v = torch.from_numpy(inp.v8).cuda()
    dv = torch.tensor([inp.descale[2]], dtype=torch.float32, device="cuda")
    return q, k, v, dv


def _oracle(inp, rows, p_mode, block_scale, causal=1):
    import oracle
    wl = inp.wl
    p = oracle.make_params(dtype="mixed", B=wl.B, Hq=wl.Hq, Hkv=wl.Hkv, N=wl.N, d_qk=wl.d_qk,
                           d_v=wl.d_v, descale=(1.0, 1.0, inp.descale[2]), p_mode=p_mode,
                           block_scale=block_scale, causal=causal)
    out, outb, lse = oracle.fwd(p, inp.q16, inp.k16, inp.v8, rows)
    return oracle.bf16_bits_to_f64(outb), out, lse


def _score_bound(inp):
    """Per row (b, h, i) of all rows: d u c max_j sum_i |q_i k_ji| over the
    visible keys, in nats."""
    import oracle
    wl = inp.wl
    q = np.abs(oracle.bf16_bits_to_f64(inp.q16))          # [B, N, Hq, d]
    k = np.abs(oracle.bf16_bits_to_f64(inp.k16))          # [B, N, Hkv, d]
    grp = wl.Hq // wl.Hkv
    c = 1.0 / np.sqrt(wl.d_qk)
    out = np.empty((wl.B, wl.Hq, wl.N))
    mask = np.tril(np.ones((wl.N, wl.N), dtype=bool))
    for b in range(wl.B):
        for h in range(wl.Hq):
            a = q[b, :, h] @ k[b, :, h // grp].T                 # sum_i |q_i||k_ji|
            out[b, h] = np.where(mask, a, 0.0).max(axis=1)
    return (wl.d_qk * 2.0 ** -24 * c * out).reshape(-1)


CASES = [
    # B, Hq, Hkv, N, d_qk, kind
    (1, 1, 1, 256, 128, "gaussian"),
    (2, 4, 2, 384, 128, "gaussian"),
    (1, 4, 2, 1024, 128, "sink"),
    (1, 2, 2, 384, 192, "gaussian"),
    (2, 4, 1, 256, 192, "activation"),
]


@pytest.mark.parametrize("mode", [(1, 1), (0, 1), (1, 0), (0, 0)], ids=["lean", "exact", "lean_nobs", "exact_nobs"])
@pytest.mark.parametrize("case", CASES, ids=[f"{c[5]}-{c[0]}x{c[1]}x{c[2]}x{c[3]}x{c[4]}" for c in CASES])
def test_mixed_all_rows(lib, case, mode):
    import torch
    wl = S.Workload("mx", *case[:5], 128, kind=case[5])
    inp = S.make_inputs(wl, seed=21, fp8=True, bf16=True)
    q, k, v, dv = _dev(inp)
    out, lse = lib.attention_bf16qk_fp8pv(q, k, v, dv, p_mode=mode[0], block_scale=mode[1],
                                          return_lse=True)
    torch.cuda.synchronize()
    rows = np.arange(wl.B * wl.Hq * wl.N)
    got = P.gather_rows(out, wl, rows)
    ref_b, ref, ref_lse = _oracle(inp, rows, *mode)
    rel = np.linalg.norm(got - ref_b) / np.linalg.norm(ref_b)
    assert rel <= STRICT_REL_L2, rel
    # LSE: the scores come from BF16 operands accumulated in FP32, whose error
    # is at most d u c sum_i |q_i k_i| per key (u = 2^-24), and the LSE moves
    # by at most the largest score error of its row.  Beyond that bound the
    # FP8 limits apply (tests/test_gpu_lse.py: 2e-2 worst row, 5e-4 RMS).
    lse_g = lse.reshape(-1).cpu().numpy().astype(np.float64)[rows]
    excess = np.maximum(np.abs(lse_g - ref_lse) - _score_bound(inp), 0.0)
    assert np.max(excess) < 2e-2 and np.sqrt(np.mean(excess ** 2)) < 5e-4, (
        np.max(excess), np.sqrt(np.mean(excess ** 2)))


def test_mixed_noncausal(lib):
    import torch
    wl = S.Workload("mxn", 1, 2, 1, 512, 128, 128)
    inp = S.make_inputs(wl, seed=22, fp8=True, bf16=True)
    q, k, v, dv = _dev(inp)
    out = lib.attention_bf16qk_fp8pv(q, k, v, dv, causal=0)
    torch.cuda.synchronize()
    rows = np.arange(wl.B * wl.Hq * wl.N)
    ref_b, _, _ = _oracle(inp, rows, 1, 1, causal=0)
    got = P.gather_rows(out, wl, rows)
    assert np.linalg.norm(got - ref_b) / np.linalg.norm(ref_b) <= STRICT_REL_L2


@pytest.mark.parametrize("name", ["d128", "mla"])
def test_mixed_full_size_sampled(lib, name):
    import torch
    wl = S.WORKLOADS[name]
    inp = S.make_inputs(wl, fp8=True, bf16=True)
    q, k, v, dv = _dev(inp)
    out = lib.attention_bf16qk_fp8pv(q, k, v, dv)
    torch.cuda.synchronize()
    rows = S.sample_rows(wl, per_head=64)
    ref_b, _, _ = _oracle(inp, rows, 1, 1)
    got = P.gather_rows(out, wl, rows)
    rel = np.linalg.norm(got - ref_b) / np.linalg.norm(ref_b)
    print(name, "rel-L2 vs oracle", rel)
    assert rel <= STRICT_REL_L2


def test_mixed_removes_most_input_error(lib):
    """Sec. VII: keeping QK^T in BF16 removes most of the input error.  On
    activation-like inputs (outlier channels shared by q and k), the error
    against fp64 attention on the BF16 inputs must be well below all-FP8's."""
    import torch
    import oracle
    wl = S.Workload("ie", 1, 4, 1, 1024, 128, 128, kind="activation")
    inp = S.make_inputs(wl, seed=23, fp8=True, bf16=True)
    rows = np.arange(wl.B * wl.Hq * wl.N)
    p64 = oracle.make_params(dtype="bf16", B=1, Hq=4, Hkv=1, N=1024, d_qk=128, d_v=128)
    exact = oracle.attn_fp64(p64, inp.q16, inp.k16, inp.v16, rows)[0]
    q, k, v, dv = _dev(inp)
    mixed = P.gather_rows(lib.attention_bf16qk_fp8pv(q, k, v, dv), wl, rows)
    fp8 = P.gather_rows(P.gpu_run(inp, "lean"), wl, rows)
    torch.cuda.synchronize()
    e_mixed = np.linalg.norm(mixed - exact) / np.linalg.norm(exact)
    e_fp8 = np.linalg.norm(fp8 - exact) / np.linalg.norm(exact)
    print("rel-L2 vs fp64 on BF16 inputs: all-FP8", e_fp8, "BF16 QK / FP8 PV", e_mixed)
    assert e_mixed < 0.5 * e_fp8
