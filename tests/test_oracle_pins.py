"""Pins for the CPU oracle, each against something other than the oracle itself.

  * e4m3 decode: every byte against torch's float8_e4m3fn, plus values fixed by the format.
  * bf16 rounding: torch's fp32 -> bf16 (single rounding) on fp32-exact values; hand-built
    double-rounding traps, subnormals and overflow fixed by the format.
  * convolution: brute force on tiny inputs through an independent formulation (explicit zero
    padding + strided slices + einsum); torch.nn.functional.conv3d in fp64 (exact sums, so bitwise
    equal); 1x1x1 filter == GEMM; delta filter == shifted copy; all-ones input == partial sums of
    the filter over the in-bounds taps; power-of-two scales.
  * padded-row alias predictor: the figures the subject page prints.
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import alias
from conftest import read_golden
from fp8_implicit_gemm_gb300 import synth

ONE = 0x38  # e4m3 1.0


# ------------------------------------------------------------------------------------------ e4m3
def test_e4m3_decode_all_bytes_match_torch():
    b = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(b)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zero is kept
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_e4m3_decode_format_values():
    d = oracle.e4m3_decode(np.array([0x38, 0x7E, 0xFE, 0x01, 0x07, 0x08, 0x40, 0x30, 0x00],
                                    dtype=np.uint8))
    assert list(d) == [1.0, 448.0, -448.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 2.0, 0.5, 0.0]
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)                         # monotone over the positive codes
    assert np.all(pos * 512 == np.round(pos * 512))         # integer multiples of 2^-9


# ------------------------------------------------------------------------------------------ bf16
def _torch_bf16_bits_from_f32(v):
    t = torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_rne_matches_torch_on_fp32_values():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 30, 20000))).astype(np.float32)
    # exact ties (low 16 bits == 0x8000) with both parities of the kept bit
    ties = (rng.integers(0, 2 ** 31, 4000, dtype=np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    v = np.concatenate([v, ties.view(np.float32)])
    v = v[np.isfinite(v)]
    assert np.array_equal(oracle.bf16_rne(v.astype(np.float64)), _torch_bf16_bits_from_f32(v))


def test_bf16_rne_single_rounding_from_double():
    # 1 + 2^-8 is the midpoint between bf16 1.0 and 1 + 2^-7; a double just above it must round up
    # even though rounding to fp32 first would land on the tie and then round to even (down).
    above = 1.0 + 2.0 ** -8 + 2.0 ** -40
    below = 1.0 + 2.0 ** -8 - 2.0 ** -40
    tie_even = 1.0 + 2.0 ** -8
    tie_odd = 1.0 + 3 * 2.0 ** -8       # midpoint between 1+2^-7 (odd) and 1+2^-6 (even)
    got = oracle.bf16_rne([above, below, tie_even, tie_odd, -above])
    assert list(got) == [0x3F81, 0x3F80, 0x3F80, 0x3F82, 0xBF81]


def test_bf16_rne_edges():
    got = oracle.bf16_rne([0.0, -0.0, 2.0 ** -133, 2.0 ** -134, 1.5 * 2.0 ** -133, 2.0 ** -126,
                           float.fromhex("0x1.fep127"), float.fromhex("0x1.ffp127"), float("inf"), -float("inf")])
    assert list(got) == [0x0000, 0x8000, 0x0001, 0x0000, 0x0002, 0x0080,
                         0x7F7F, 0x7F80, 0x7F80, 0xFF80]
    assert oracle.bf16_rne([float("nan")])[0] & 0x7F80 == 0x7F80


# ------------------------------------------------------------------------------ convolution sums
def _decoded(b):
    return oracle.e4m3_decode(np.arange(256, dtype=np.uint8))[np.asarray(b, dtype=np.uint8)]


def _independent_sum(x, w, stride, pad):
    """Zero-pad explicitly, then add one strided slice per tap (einsum over channels)."""
    X, Wt = _decoded(x), _decoded(w)
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


def _rand_bytes(rng, shape):
    b = rng.integers(0, 256, size=shape, dtype=np.uint8)
    b[(b & 0x7F) == 0x7F] = 0x7E  # no NaN codes
    return b


def test_tiny_brute_force_against_padded_slices():
    rng = np.random.default_rng(11)
    for trial in range(60):
        N, C, K = rng.integers(1, 3), rng.integers(1, 4), rng.integers(1, 3)
        T, R, S = (int(v) for v in rng.integers(1, 4, 3))
        stride = tuple(int(v) for v in rng.integers(1, 3, 3))
        pad = tuple(int(v) for v in rng.integers(0, 3, 3))
        D, H, W = (int(max(v, k - 2 * p)) for v, k, p in
                   zip(rng.integers(1, 5, 3), (T, R, S), pad))
        x = _rand_bytes(rng, (N, C, D, H, W))
        w = _rand_bytes(rng, (K, C, T, R, S))
        ysum, y64, yb = oracle.conv3d_fp8(x, w, 1.0, 1.0, stride, pad, want_sum=True)
        ref = _independent_sum(x, w, stride, pad)
        assert ysum.shape == ref.shape, (trial, ysum.shape, ref.shape)
        assert np.array_equal(ysum, ref), trial
        assert np.array_equal(y64, ref)


@pytest.mark.parametrize("cfg", [0, 3])
def test_full_config_matches_torch_conv3d_fp64(cfg):
    """Sums are exact in fp64 in any order, so torch's fp64 conv3d must agree bit for bit."""
    shp = synth.CONFIGS[cfg]
    inp = synth.make_config_inputs(cfg)
    x, w = inp["x"].numpy(), inp["w"].numpy()
    ysum, y64, yb = oracle.conv3d_fp8(x, w, inp["sx"], inp["sw"], shp.stride, shp.pad,
                                      want_sum=True)
    X = torch.from_numpy(_decoded(x))
    Wt = torch.from_numpy(_decoded(w))
    ref = F.conv3d(X, Wt, stride=shp.stride, padding=shp.pad).numpy()
    assert np.array_equal(ysum, ref)
    assert np.array_equal(y64, (np.float64(inp["sx"]) * np.float64(inp["sw"])) * ref)


def test_tiny_matches_torch_conv3d_fp64_all_strides_pads():
    rng = np.random.default_rng(5)
    for stride, pad in itertools.product([1, 2, 3], [0, 1, 2]):
        x = _rand_bytes(rng, (2, 3, 5, 6, 7))
        w = _rand_bytes(rng, (4, 3, 3, 3, 3))
        ysum, _, _ = oracle.conv3d_fp8(x, w, 1.0, 1.0, stride, pad, want_sum=True)
        ref = F.conv3d(torch.from_numpy(_decoded(x)), torch.from_numpy(_decoded(w)),
                       stride=stride, padding=pad).numpy()
        assert np.array_equal(ysum, ref), (stride, pad)


def test_out_dims_match_torch():
    for D, k, s, p in itertools.product([1, 4, 9, 16], [1, 2, 3], [1, 2, 3], [0, 1, 2]):
        if D + 2 * p < k:
            continue
        ref = F.conv3d(torch.zeros(1, 1, D, 1, 1), torch.zeros(1, 1, k, 1, 1),
                       stride=(s, 1, 1), padding=(p, 0, 0)).shape[2]
        assert oracle.out_dims(D, 1, 1, k, 1, 1, (s, 1, 1), (p, 0, 0))[0] == ref


def test_1x1x1_filter_is_a_gemm():
    rng = np.random.default_rng(3)
    x = _rand_bytes(rng, (2, 48, 3, 4, 5))
    w = _rand_bytes(rng, (32, 48, 1, 1, 1))
    ysum, _, _ = oracle.conv3d_fp8(x, w, 1.0, 1.0, 1, 0, want_sum=True)
    X = _decoded(x).reshape(2, 48, -1)
    Wm = _decoded(w).reshape(32, 48)
    ref = np.stack([Wm @ X[n] for n in range(2)]).reshape(ysum.shape)
    assert np.array_equal(ysum, ref)


@pytest.mark.parametrize("stride", [1, 2])
def test_delta_filter_is_a_shifted_copy(stride):
    rng = np.random.default_rng(9)
    C = 4
    x = _rand_bytes(rng, (1, C, 5, 6, 7))
    X = _decoded(x)
    for t0, r0, s0 in itertools.product(range(3), repeat=3):
        w = np.zeros((C, C, 3, 3, 3), np.uint8)
        for c in range(C):
            w[c, c, t0, r0, s0] = ONE
        ysum, _, _ = oracle.conv3d_fp8(x, w, 1.0, 1.0, stride, 1, want_sum=True)
        _, K, Do, Ho, Wo = ysum.shape
        for od, oh, ow in itertools.product(range(Do), range(Ho), range(Wo)):
            d, h, ww = od * stride + t0 - 1, oh * stride + r0 - 1, ow * stride + s0 - 1
            inside = 0 <= d < 5 and 0 <= h < 6 and 0 <= ww < 7
            exp = X[0, :, d, h, ww] if inside else np.zeros(C)
            assert np.array_equal(ysum[0, :, od, oh, ow], exp), (t0, r0, s0, od, oh, ow)


def test_all_ones_input_gives_partial_filter_sums():
    rng = np.random.default_rng(4)
    C, K, D, H, W = 3, 2, 4, 5, 6
    x = np.full((1, C, D, H, W), ONE, np.uint8)
    w = _rand_bytes(rng, (K, C, 3, 3, 3))
    ysum, _, _ = oracle.conv3d_fp8(x, w, 1.0, 1.0, 1, 1, want_sum=True)
    Wc = _decoded(w).sum(axis=1)                    # [K, 3, 3, 3]: channels summed
    total = Wc.sum(axis=(1, 2, 3))
    # interior: every tap in bounds
    assert np.array_equal(ysum[0, :, 1, 1, 1], total)
    assert np.array_equal(ysum[0, :, 2, 3, 4], total)
    # corner (0,0,0): the 8 taps t,r,s in {1,2}
    assert np.array_equal(ysum[0, :, 0, 0, 0], Wc[:, 1:, 1:, 1:].sum(axis=(1, 2, 3)))
    # opposite corner: the 8 taps t,r,s in {0,1}
    assert np.array_equal(ysum[0, :, D - 1, H - 1, W - 1], Wc[:, :2, :2, :2].sum(axis=(1, 2, 3)))
    # edge (0,0,interior): 12 taps
    assert np.array_equal(ysum[0, :, 0, 0, 2], Wc[:, 1:, 1:, :].sum(axis=(1, 2, 3)))
    # face (0,interior,interior): 18 taps
    assert np.array_equal(ysum[0, :, 0, 2, 2], Wc[:, 1:, :, :].sum(axis=(1, 2, 3)))


def test_scales_power_of_two_are_exact_and_rounding_is_bf16():
    rng = np.random.default_rng(21)
    x = _rand_bytes(rng, (1, 4, 3, 4, 5))
    w = _rand_bytes(rng, (3, 4, 3, 3, 3))
    ysum, y64, yb = oracle.conv3d_fp8(x, w, 0.5, 0.125, 1, 1, want_sum=True)
    assert np.array_equal(y64, ysum / 16.0)
    ref_bits = _torch_bf16_bits_from_f32(y64.astype(np.float32))
    exact_in_f32 = y64.astype(np.float32).astype(np.float64) == y64
    assert np.array_equal(yb[exact_in_f32], ref_bits[exact_in_f32])


def test_points_agree_with_full_output():
    shp = synth.CONFIGS[0]
    inp = synth.make_config_inputs(0)
    y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                shp.stride, shp.pad)
    rng = np.random.default_rng(0)
    idx = rng.integers(0, y64.size, 500)
    p64, pb = oracle.conv3d_fp8_points(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                       idx, shp.stride, shp.pad)
    assert np.array_equal(p64, y64.ravel()[idx])
    assert np.array_equal(pb, yb.ravel()[idx])


def test_nan_input_byte_is_rejected():
    x = np.full((1, 1, 2, 2, 2), ONE, np.uint8)
    w = np.full((1, 1, 1, 1, 1), ONE, np.uint8)
    x[0, 0, 1, 1, 1] = 0x7F
    with pytest.raises(ValueError):
        oracle.conv3d_fp8(x, w, 1.0, 1.0, 1, 0)
    with pytest.raises(IndexError):
        oracle.conv3d_fp8_points(w.repeat(2, axis=2), w, 1.0, 1.0, [5], 1, 0)


# ------------------------------------------------------------------------ alias predictor (page)
def test_alias_predictor_reproduces_page_figures():
    g = read_golden("p1_padded_row_alias.txt")
    N, K = int(g["N"]), int(g["K"])
    Do, Ho, Wo = oracle.out_dims(int(g["D"]), int(g["H"]), int(g["W"]), 3, 3, 3,
                                 int(g["stride"]), int(g["pad"]))
    dhw = Do * Ho * Wo
    npq = N * dhw
    tile = int(g["tile_m"])
    assert npq == int(g["npq"])
    assert alias.grid_m(npq, tile) == int(g["grid_m"])
    assert alias.padded_rows(npq, tile) == int(g["padded_rows"])
    assert int(dhw == npq) == int(g["dhw_equals_npq"])
    offs = alias.clobberable_offsets(N, K, dhw, tile)
    assert len(offs) == int(g["clobbered_offsets"])
    assert round(100.0 * len(offs) / (N * K * dhw), 2) == float(g["clobbered_percent"])
    # padded row 288 of column 0 is the live row 0 of column 1
    assert int(g["example_alias_offset"]) in offs
    assert 0 * dhw + npq == 1 * dhw + 0


def test_alias_predictor_other_configs():
    # n > 1 or padded-row-free shapes expose nothing; the large unaligned layer does
    assert alias.clobberable_offsets(2, 128, 1920, 128) == set()
    assert alias.clobberable_offsets(1, 128, 65536, 128) == set()
    offs = alias.clobberable_offsets(1, 256, 244800, 128)
    assert len(offs) == 64 * 255
