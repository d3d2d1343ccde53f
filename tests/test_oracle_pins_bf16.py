"""Pins for the BF16-input twin of the CPU oracle, each against something other than the oracle.

  * bfloat16 decode: all 65536 bit patterns against torch's bfloat16, plus values fixed by the
    format.
  * convolution: brute force on tiny inputs through an independent formulation (explicit zero
    padding + strided slices + einsum on torch-decoded values), on values whose products and sums
    are exact in fp64, so the comparison is bitwise; torch.nn.functional.conv3d in fp64 on a
    seeded workload (sums rounded in a different order: equal within the recursive-summation
    bound); 1x1x1 filter == GEMM; delta filter == shifted copy; all-ones input == partial sums of
    the filter over the in-bounds taps; infinite and NaN inputs rejected.
"""
import itertools

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from fp8_implicit_gemm_gb300 import synth

ONE = 0x3F80  # bfloat16 1.0


def _torch_decode(bits) -> np.ndarray:
    """Value of bfloat16 bit patterns through torch (independent of the oracle's decoder)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double().numpy()


def _to_bits(values) -> np.ndarray:
    """bfloat16 bit patterns of values that bfloat16 holds exactly (checked)."""
    t = torch.from_numpy(np.asarray(values, dtype=np.float64)).to(torch.bfloat16)
    assert np.array_equal(t.double().numpy(), np.asarray(values, dtype=np.float64))
    return t.view(torch.int16).numpy().view(np.uint16)


def _dyadic(rng, shape, lo=-8, hi=8, e=3):
    """Small integers times 2^j (|j| <= e): products and sums of a few hundred stay exact."""
    m = rng.integers(lo, hi + 1, size=shape).astype(np.float64)
    j = rng.integers(-e, e + 1, size=shape)
    return _to_bits(np.ldexp(m, j))


# ------------------------------------------------------------------------------------- decoding
def test_bf16_decode_all_patterns_match_torch():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_decode(b)
    ref = _torch_decode(b)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_format_values():
    cases = {0x3F80: 1.0, 0x4000: 2.0, 0xBF80: -1.0, 0x3F00: 0.5, 0x3FC0: 1.5,
             0x0001: 2.0 ** -133, 0x007F: 127 * 2.0 ** -133, 0x0080: 2.0 ** -126,
             0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127, 0x0000: 0.0, 0x7F80: np.inf, 0xFF80: -np.inf}
    for bits, v in cases.items():
        assert oracle.bf16_decode(np.array([bits], np.uint16))[0] == v, hex(bits)
    assert np.isnan(oracle.bf16_decode(np.array([0x7FC0, 0xFFC1], np.uint16))).all()


# --------------------------------------------------------------------------------- convolution
def _independent_sum(x, w, stride, pad):
    """Zero-pad explicitly, then add one strided slice per tap (einsum over channels)."""
    X, Wt = _torch_decode(x), _torch_decode(w)
    N, C, D, H, W = X.shape
    K, _, T, R, S = Wt.shape
    (sd, sh, sw), (pd, ph, pw) = stride, pad
    Xp = np.pad(X, ((0, 0), (0, 0), (pd, pd), (ph, ph), (pw, pw)))
    Do, Ho, Wo = (D + 2 * pd - T) // sd + 1, (H + 2 * ph - R) // sh + 1, (W + 2 * pw - S) // sw + 1
    out = np.zeros((N, K, Do, Ho, Wo))
    for t, r, s in itertools.product(range(T), range(R), range(S)):
        sl = Xp[:, :, t:t + sd * (Do - 1) + 1:sd, r:r + sh * (Ho - 1) + 1:sh,
                s:s + sw * (Wo - 1) + 1:sw]
        out += np.einsum("ncdhw,kc->nkdhw", sl, Wt[:, :, t, r, s])
    return out


def test_tiny_brute_force_against_padded_slices():
    rng = np.random.default_rng(21)
    for trial in range(60):
        N, C, K = rng.integers(1, 3), rng.integers(1, 4), rng.integers(1, 3)
        T, R, S = (int(v) for v in rng.integers(1, 4, 3))
        stride = tuple(int(v) for v in rng.integers(1, 3, 3))
        pad = tuple(int(v) for v in rng.integers(0, 3, 3))
        D, H, W = (int(max(v, k - 2 * p)) for v, k, p in
                   zip(rng.integers(1, 5, 3), (T, R, S), pad))
        x = _dyadic(rng, (N, C, D, H, W))
        w = _dyadic(rng, (K, C, T, R, S))
        y64, yb = oracle.conv3d_bf16(x, w, stride, pad)
        ref = _independent_sum(x, w, stride, pad)
        assert y64.shape == ref.shape, trial
        assert np.array_equal(y64, ref), trial
        # the BF16 output is the single rounding of the exact value (torch's double -> bf16)
        refb = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(yb, refb), trial


def test_seeded_workload_matches_torch_conv3d_fp64():
    """Random N(0,1) bfloat16 inputs: fp64 sums in two orders agree within the summation bound."""
    shp = synth.CONFIGS[0]
    inp = synth.make_config_inputs_bf16(0)
    x, w = synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["w"])
    y64, yb = oracle.conv3d_bf16(x, w, shp.stride, shp.pad)
    X = inp["x"].double()
    Wt = inp["w"].double()
    ref = F.conv3d(X, Wt, stride=shp.stride, padding=shp.pad).numpy()
    absum = F.conv3d(X.abs(), Wt.abs(), stride=shp.stride, padding=shp.pad).numpy()
    n = shp.C * shp.T * shp.R * shp.S
    assert np.all(np.abs(y64 - ref) <= 2 * n * 2.0 ** -53 * absum)
    # BF16 bits agree wherever the value is not within that bound of a rounding boundary
    refb = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.mean(yb == refb) > 0.9999


def test_1x1x1_filter_is_a_gemm():
    rng = np.random.default_rng(23)
    x = _dyadic(rng, (2, 48, 3, 4, 5))
    w = _dyadic(rng, (32, 48, 1, 1, 1))
    y64, _ = oracle.conv3d_bf16(x, w, 1, 0)
    X = _torch_decode(x).reshape(2, 48, -1)
    Wm = _torch_decode(w).reshape(32, 48)
    ref = np.stack([Wm @ X[n] for n in range(2)]).reshape(y64.shape)
    assert np.array_equal(y64, ref)


@pytest.mark.parametrize("stride", [1, 2])
def test_delta_filter_is_a_shifted_copy(stride):
    rng = np.random.default_rng(29)
    C = 4
    x = (torch.from_numpy(rng.standard_normal((1, C, 5, 6, 7))).to(torch.bfloat16)
         .view(torch.int16).numpy().view(np.uint16))
    X = _torch_decode(x)
    for t0, r0, s0 in itertools.product(range(3), repeat=3):
        w = np.zeros((C, C, 3, 3, 3), np.uint16)
        for c in range(C):
            w[c, c, t0, r0, s0] = ONE
        y64, yb = oracle.conv3d_bf16(x, w, stride, 1)
        _, K, Do, Ho, Wo = y64.shape
        for od, oh, ow in itertools.product(range(Do), range(Ho), range(Wo)):
            d, h, ww = od * stride + t0 - 1, oh * stride + r0 - 1, ow * stride + s0 - 1
            inside = 0 <= d < 5 and 0 <= h < 6 and 0 <= ww < 7
            exp = X[0, :, d, h, ww] if inside else np.zeros(C)
            assert np.array_equal(y64[0, :, od, oh, ow], exp), (t0, r0, s0, od, oh, ow)
            # one exact term: the BF16 output is the input's own bit pattern (or +0)
            expb = x[0, :, d, h, ww] if inside else np.zeros(C, np.uint16)
            assert np.array_equal(yb[0, :, od, oh, ow], expb)


def test_all_ones_input_gives_partial_filter_sums():
    rng = np.random.default_rng(31)
    C, K, D, H, W = 3, 2, 4, 5, 6
    x = np.full((1, C, D, H, W), ONE, np.uint16)
    w = _dyadic(rng, (K, C, 3, 3, 3))
    y64, _ = oracle.conv3d_bf16(x, w, 1, 1)
    Wc = _torch_decode(w).sum(axis=1)
    total = Wc.sum(axis=(1, 2, 3))
    assert np.array_equal(y64[0, :, 1, 1, 1], total)
    assert np.array_equal(y64[0, :, 2, 3, 4], total)
    assert np.array_equal(y64[0, :, 0, 0, 0], Wc[:, 1:, 1:, 1:].sum(axis=(1, 2, 3)))
    assert np.array_equal(y64[0, :, D - 1, H - 1, W - 1], Wc[:, :2, :2, :2].sum(axis=(1, 2, 3)))
    assert np.array_equal(y64[0, :, 0, 0, 2], Wc[:, 1:, 1:, :].sum(axis=(1, 2, 3)))
    assert np.array_equal(y64[0, :, 0, 2, 2], Wc[:, 1:, :, :].sum(axis=(1, 2, 3)))


def test_points_agree_with_full_output():
    shp = synth.ConvShape(2, 16, 3, 5, 6, 24, stride=(1, 2, 1), pad=(1, 0, 2))
    inp = synth.make_inputs_bf16(shp, 3)
    x, w = synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["w"])
    y64, yb = oracle.conv3d_bf16(x, w, shp.stride, shp.pad)
    idx = np.random.default_rng(0).integers(0, y64.size, 500)
    p64, pb = oracle.conv3d_bf16_points(x, w, idx, shp.stride, shp.pad)
    assert np.array_equal(p64, y64.ravel()[idx]) and np.array_equal(pb, yb.ravel()[idx])
    with pytest.raises(IndexError):
        oracle.conv3d_bf16_points(x, w, np.array([y64.size]), shp.stride, shp.pad)


@pytest.mark.parametrize("bad", [0x7F80, 0xFF80, 0x7FC0])
def test_infinite_or_nan_input_is_rejected(bad):
    x = np.full((1, 2, 3, 3, 3), ONE, np.uint16)
    w = np.full((2, 2, 1, 1, 1), ONE, np.uint16)
    x[0, 1, 1, 1, 1] = bad
    with pytest.raises(ValueError):
        oracle.conv3d_bf16(x, w, 1, 0)
