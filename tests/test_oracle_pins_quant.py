"""Pins for the quantiser oracle (oracle/quantize.py), each against something other than itself.

  * e4m3 rounding: every finite grid value maps to its own code and decodes back (through the
    convolution oracle's decoder, pinned on its own); every midpoint between neighbours rounds to
    the even code; 10^6 random fp32 values agree with torch's float8_e4m3fn cast.
  * fp32 division and the scale: equal to the exactly rounded rational quotient (Python fractions)
    on random and near-tie operands, which pins the float64-then-fp32 argument.
  * quantise: the largest magnitude lands on +-448 exactly, an all-zero tensor gets scale 1, and
    the bytes and scale equal the harness quantiser's (torch) on the workloads' tensors.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import quantize as Q
from fp8_implicit_gemm_gb300 import synth


def _round_to_f32(fr: Fraction) -> np.float32:
    """Exactly rounded (to nearest, ties to even) fp32 value of a rational, normal range."""
    if fr == 0:
        return np.float32(0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (e - 23)       # fp32 spacing in the binade [2^e, 2^(e+1))
    k = a / q
    fl = k.numerator // k.denominator
    rem = k - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return np.float32(sign * float(fl * q))


def _grid():
    """All finite non-negative e4m3 values with their codes, from the format definition."""
    vals, codes = [], []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (8 + m) * 2.0 ** (e - 10))
        codes.append(code)
    return np.array(vals), np.array(codes, dtype=np.uint8)


def test_grid_values_map_to_their_codes_and_back():
    vals, codes = _grid()
    for sgn, bit in ((1.0, 0), (-1.0, 0x80)):
        got = Q.e4m3_rne(sgn * vals)
        exp = codes | bit
        if sgn < 0:
            exp[0] = 0x80  # -0
        assert np.array_equal(got, exp)
    assert np.array_equal(oracle.e4m3_decode(Q.e4m3_rne(vals)), vals)


def test_midpoints_round_to_even():
    vals, codes = _grid()
    mids = (vals[:-1] + vals[1:]) / 2
    got = Q.e4m3_rne(mids)
    lo, hi = codes[:-1], codes[1:]
    exp = np.where(lo % 2 == 0, lo, hi)  # the even mantissa (codes of neighbours differ by one)
    assert np.array_equal(got, exp)
    # just below / above a midpoint go to the nearer neighbour
    assert np.array_equal(Q.e4m3_rne(np.nextafter(mids, 0)), lo)
    assert np.array_equal(Q.e4m3_rne(np.nextafter(mids, 1000)), hi)


def test_rounding_matches_torch_cast_on_random_values():
    rng = np.random.default_rng(3)
    mag = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 1_000_000))
    v = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(Q.e4m3_rne(v), ref)


def test_fp32_division_is_the_exactly_rounded_quotient():
    rng = np.random.default_rng(5)
    for _ in range(3000):
        a = np.float32(rng.standard_normal() * 10 ** rng.uniform(-3, 3))
        b = np.float32(abs(rng.standard_normal()) * 10 ** rng.uniform(-3, 1) + 1e-6)
        assert Q.fp32_div(a, b) == _round_to_f32(Fraction(float(a)) / Fraction(float(b)))
    # operands whose quotient sits near fp32 ties: b = 3, 7, 448 and significands near 1.5
    for b in (3.0, 7.0, 448.0):
        for k in range(2000):
            a = np.float32((1 << 23) + 3 * k) * np.float32(2.0 ** -20)
            assert Q.fp32_div(a, b) == _round_to_f32(Fraction(float(a)) / Fraction(b))


def test_division_differs_from_a_reciprocal_multiply_where_it_should():
    """A reciprocal multiply in fp32 (v * fp32(1/s)) is a plausible slip: find operand pairs where
    it differs from the true quotient and check that the oracle gives the exactly rounded one."""
    rng = np.random.default_rng(11)
    a = rng.uniform(1, 2, 200_000).astype(np.float32)
    b = rng.uniform(1, 2, 200_000).astype(np.float32)
    via_recip = a * (np.float32(1.0) / b)  # fp32 arithmetic throughout
    cand = np.nonzero(via_recip != Q.fp32_div(a, b))[0]
    assert cand.size > 0
    for i in cand[:200]:
        exact = _round_to_f32(Fraction(float(a[i])) / Fraction(float(b[i])))
        assert Q.fp32_div(a[i], b[i]) == exact
        assert via_recip[i] != exact


def test_scale_is_the_exactly_rounded_amax_over_448():
    rng = np.random.default_rng(7)
    for _ in range(3000):
        amax = np.float32(abs(rng.standard_normal()) * 10 ** rng.uniform(-4, 4))
        assert Q.scale_of(amax) == _round_to_f32(Fraction(float(amax)) / 448)
    assert Q.scale_of(np.float32(448.0)) == np.float32(1.0)
    assert Q.scale_of(np.float32(0.0)) == np.float32(1.0)


@pytest.mark.parametrize("seed", range(5))
def test_largest_magnitude_lands_on_448(seed):
    rng = np.random.default_rng(seed)
    v = (rng.standard_normal(10000) * 10 ** rng.uniform(-3, 3)).astype(np.float32)
    q, s = Q.quantize(v)
    i = int(np.argmax(np.abs(v)))
    assert q[i] == (0xFE if v[i] < 0 else 0x7E)
    assert not np.any((q & 0x7F) == 0x7F)  # never a NaN code


def test_all_zero_tensor():
    q, s = Q.quantize(np.zeros(100, np.float32))
    assert s == np.float32(1.0) and not q.any()


@pytest.mark.parametrize("cfg", [0, 1, 3])
def test_matches_the_harness_quantiser(cfg):
    """synth's quantiser (torch, used to make every workload's inputs) gives the same bytes."""
    shape = synth.CONFIGS[cfg]
    g = torch.Generator().manual_seed(123 + cfg)
    v = torch.randn((shape.N, shape.C, shape.D, shape.H, shape.W), generator=g)
    tq, ts = synth.quantize_e4m3(v)
    q, s = Q.quantize(v.numpy())
    assert np.float32(ts) == s
    assert np.array_equal(q.reshape(tq.shape), tq.numpy())
    idx = np.arange(0, v.numel(), 97)
    assert np.array_equal(Q.quantize_points(v.numpy(), idx, s), q.ravel()[idx])
