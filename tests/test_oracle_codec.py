"""Pins of the oracle's number formats and probability codes (CPU only).

Each test checks the oracle against something other than itself: values the
paper prints (tests/golden/paper_constants.json), exhaustive enumeration,
an exact-rational brute force, or PyTorch's own conversions.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import brute_force as bf


def test_e4m3_printed_codes(golden):
    for code, val in golden["e4m3_printed_codes"]["pairs"]:
        assert oracle.e4m3_decode(code) == val
        assert oracle.e4m3_encode(val) == code


def test_e4m3_range_constants(golden):
    assert oracle.e4m3_decode(0x7E) == golden["e4m3_max_finite"]["value"]
    assert oracle.e4m3_decode(8) == golden["e4m3_smallest_normal"]["value"]
    assert oracle.e4m3_decode(1) == golden["e4m3_subnormal_spacing"]["value"]
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))
    lo = golden["e4m3_rounds_to_zero_below"]["value"]
    assert oracle.e4m3_encode(lo * 0.999) == 0
    assert oracle.e4m3_encode(lo) == 0          # the tie goes to the even code 0
    assert oracle.e4m3_encode(lo * 1.001) == 1
    assert oracle.e4m3_encode(1e6) == 0x7E and oracle.e4m3_encode(-1e6) == 0xFE


def test_e4m3_decode_matches_bitfields_and_torch():
    ours = oracle.e4m3_decode_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(ours[fin], bf.e4m3_values()[fin])


def test_e4m3_roundtrip_every_code():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c


def test_e4m3_midpoints_round_to_even():
    vals = bf.e4m3_values()[:127]
    for c in range(126):
        mid = 0.5 * (vals[c] + vals[c + 1])
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == want, c
        assert bf.e4m3_encode(mid) == want
        assert oracle.e4m3_encode(-mid) == 0x80 | want


def test_e4m3_encode_vs_enumeration_and_torch():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.uniform(-4, 2.5, 3000),
                        rng.uniform(-460, 460, 500)])
    ours = np.array([oracle.e4m3_encode(v) for v in x])
    enum = np.array([bf.e4m3_encode(v) for v in x])
    assert np.array_equal(ours, enum)
    # torch's cast rounds to nearest even and overflows to NaN beyond 464
    xs = x[np.abs(x) < 464]
    tor = torch.from_numpy(xs.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours32 = np.array([oracle.e4m3_encode(float(np.float32(v))) for v in xs])
    assert np.array_equal(ours32, tor)


def test_bf16_encode_vs_rational_and_torch():
    rng = np.random.default_rng(6)
    x = rng.standard_normal(2000) * 10.0 ** rng.uniform(-30, 30, 2000)
    for v in x:
        assert oracle.bf16_decode(oracle.bf16_encode(v)) == bf.bf16_round(v)
    x32 = x.astype(np.float32)
    tor = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = np.array([oracle.bf16_encode(float(v)) for v in x32], dtype=np.uint16)
    assert np.array_equal(ours, tor)
    # ties to even: 1 + 2^-8 is halfway between 1 and 1 + 2^-7
    assert oracle.bf16_decode(oracle.bf16_encode(1.0 + 2 ** -8)) == 1.0
    assert oracle.bf16_decode(oracle.bf16_encode(1.0 + 3 * 2 ** -8)) == 1.0 + 2 ** -6


def test_lean_code_worked_values(golden):
    s, b = golden["lean_p"]["sigma"], golden["lean_p"]["beta"]
    # x = 0: y = 8*13 - 0.35 = 103.65 -> 104, the code of 2^6 (= p * 2^sigma)
    assert oracle.lean_code(0.0, s, b) == 104 == oracle.e4m3_encode(64.0)
    # one binade down: code drops by 8 (footnote 10)
    assert oracle.lean_code(-1.0, s, b) == 96
    # x = -0.5: y = 99.65 -> 100 = 48; exact: 2^5.5 = 45.25 -> 44 (code 99)
    assert oracle.lean_code(-0.5, s, b) == 100 and oracle.e4m3_decode(100) == 48.0
    assert oracle.exact_code(-0.5, s) == 99 and oracle.e4m3_decode(99) == 44.0
    assert oracle.lean_code(float("nan"), s, b) == 0
    assert oracle.lean_code(float("-inf"), s, b) == 0


def test_lean_error_bounds(golden):
    """Fig. 4 / Sec. IV-B1 bounds over the normal e4m3 range."""
    s, b = golden["lean_p"]["sigma"], golden["lean_p"]["beta"]
    us = np.linspace(-12.0, 0.0, 48001)[:-1]          # 2^(u+6) >= 2^-6: normal
    true = 2.0 ** (us + s)
    # the line through the codes: value(y) = 2^(E-7)(1 + F/8) with y = 8E + F
    lin = np.array([_code_line(oracle.lean_y(u, s, b)) for u in us])
    lin0 = np.array([_code_line(oracle.lean_y(u, s, 0.0)) for u in us])
    rounded = np.array([oracle.e4m3_decode(oracle.lean_code(u, s, b)) for u in us])
    exact = np.array([oracle.e4m3_decode(oracle.exact_code(u, s)) for u in us])
    e_pre = np.max(np.abs(lin / true - 1))
    e_nob = np.max(np.abs(lin0 / true - 1))
    e_rnd = np.max(np.abs(rounded / true - 1))
    e_ex = np.max(np.abs(exact / true - 1))
    assert 0.025 < e_pre <= golden["lean_error_before_rounding_max"]["value"]
    assert abs(e_nob - golden["lean_error_without_bias_max"]["value"]) < 0.003
    assert 0.07 < e_rnd <= golden["lean_error_after_rounding_max"]["value"]
    assert 0.055 < e_ex <= golden["exact_error_max"]["value"]


def _code_line(y):
    """Value that the e4m3 bit pattern y (read as a real number) stands for,
    interpolating linearly between codes (normal range)."""
    E = math.floor(y / 8.0)
    F = y - 8.0 * E
    return 2.0 ** (E - 7) * (1.0 + F / 8.0)


def test_underflow_depths(golden):
    s, b = golden["lean_p"]["sigma"], golden["lean_p"]["beta"]
    n_lean = golden["lean_underflow_binades"]["value"]
    n_exact = golden["exact_underflow_binades"]["value"]
    assert oracle.lean_code(-(n_lean - 0.2), s, b) >= 1
    assert oracle.lean_code(-n_lean, s, b) == 0
    assert oracle.exact_code(-(n_exact - 0.05), s) >= 1
    assert oracle.exact_code(-n_exact, s) == 0


def test_lean_subnormal_underestimate(golden):
    s, b = golden["lean_p"]["sigma"], golden["lean_p"]["beta"]
    us = np.linspace(-12.89, -12.0, 20000)           # subnormal, nonzero codes
    true = 2.0 ** (us + s)
    got = np.array([oracle.e4m3_decode(oracle.lean_code(u, s, b)) for u in us])
    assert np.all(got > 0)
    under = np.max(1 - got / true)
    assert abs(under - golden["lean_subnormal_underestimate"]["value"]) < 0.03
