"""The e4m3 quantiser on the GPU (conv3d_fp8_quantize, conv3d_fp8_run_quantize_x) against the
quantiser oracle and the convolution oracle, through the C ABI.

Quantised codes and scales must be bit-exact: both sides decide each code in fp32 (IEEE division
by the fp32 scale, then round-to-nearest-even onto the e4m3 grid). The fused run must then match
the convolution oracle fed the oracle's codes and scale, with the e4m3 path's gates.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import quantize as Q
from fp8_implicit_gemm_gb300 import capi, synth
from _gpu_common import GpuConv, bits, check_against, sample_indices

pytestmark = pytest.mark.gpu


def _gpu_quantize(v: torch.Tensor):
    dst = torch.empty(v.numel(), dtype=torch.uint8, device="cuda")
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    capi.conv3d_fp8_quantize(v, dst, scale)
    torch.cuda.synchronize()
    return dst.cpu().numpy(), np.float32(scale.item())


def _values(kind, n, seed):
    g = torch.Generator().manual_seed(seed)
    if kind == "normal":
        return torch.randn(n, generator=g)
    if kind == "wide":  # magnitudes over 2^-30 .. 2^10: subnormal codes and saturation at once
        e = torch.randint(-30, 11, (n,), generator=g).float()
        return torch.randn(n, generator=g) * torch.exp2(e)
    if kind == "zeros":
        return torch.zeros(n)
    raise ValueError(kind)


def _near_boundaries(amax: float, seed: int, ulps: int = 4) -> np.ndarray:
    """Values whose quotient by the scale of `amax` falls on, or within a few fp32 units of, each
    rounding boundary of the e4m3 grid (the midpoints between neighbouring codes, both signs):
    the cases where any shortcut for the IEEE quotient v / s (a multiply by fp32(1/s), say) can
    pick a different code."""
    s = Q.scale_of(np.float32(amax))
    grid = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    mids = (grid[:-1] + grid[1:]) / 2
    base = (mids * np.float64(s)).astype(np.float32)  # v with v / s near a midpoint
    out = [np.float32(amax)]
    for k in range(-ulps, ulps + 1):
        step = base.copy()
        for _ in range(abs(k)):
            step = np.nextafter(step, np.float32(np.inf if k > 0 else -np.inf)).astype(np.float32)
        out += [step, -step]
    rng = np.random.default_rng(seed)
    v = np.concatenate([np.atleast_1d(o) for o in out]).astype(np.float32)
    v = v[np.abs(v) <= np.float32(amax)]
    return v[rng.permutation(v.size)]


@pytest.mark.parametrize("amax", [448.0, 1.0, 3.7, 1234.567, 2.0 ** -20 * 5.3, 0.0625 * 7.1])
def test_quantize_quotients_near_code_boundaries(amax):
    # a multiply by fp32(1/s) would get up to 94 of these codes wrong; the quantiser divides,
    # and every value must get the code of the IEEE quotient
    v = _near_boundaries(amax, seed=int(amax * 1000) % 1000)
    q, s = _gpu_quantize(torch.from_numpy(v).cuda())
    ref_q, ref_s = Q.quantize(v)
    assert s == ref_s
    assert np.array_equal(q, ref_q), int(np.sum(q != ref_q))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("kind", ["normal", "wide", "zeros"])
@pytest.mark.parametrize("n", [1, 15, 16, 17, 1000, 65541])
def test_quantize_matches_oracle(n, kind, dtype):
    v = _values(kind, n, seed=n).to(dtype)
    q, s = _gpu_quantize(v.cuda())
    ref_q, ref_s = Q.quantize(v.float().numpy())
    assert s == ref_s
    assert np.array_equal(q, ref_q)


def test_quantize_signed_zeros_and_tiny_values():
    # a zero or a quotient that rounds to zero keeps its sign: -0 and tiny negatives give 0x80
    tiny = np.float32(2.0 ** -126)
    v = np.array([3.7, -0.0, 0.0, -tiny, tiny, -1e-30, 1e-30, -2.0 ** -140, 2.0 ** -140,
                  -1e-12, 1e-12], dtype=np.float32)
    q, s = _gpu_quantize(torch.from_numpy(v).cuda())
    ref_q, ref_s = Q.quantize(v)
    assert s == ref_s and ref_q[1] == 0x80
    assert np.array_equal(q, ref_q), [hex(a) for a in q]


@pytest.mark.parametrize("seed", range(8))
def test_quantize_dense_runs_of_consecutive_values(seed):
    # runs of consecutive fp32 values at several magnitudes under a random scale: every quotient
    # (not only those near a code boundary) must give the IEEE quotient's code
    rng = np.random.default_rng(700 + seed)
    amax = np.float32(rng.uniform(1.0, 2.0) * 2.0 ** rng.integers(-20, 11))
    runs = [np.array([amax], dtype=np.float32)]
    for frac in (1.0, 0.5, 2.0 ** -5, 2.0 ** -12, 2.0 ** -17):
        start = np.float32(amax * frac * rng.uniform(0.5, 1.0))
        run = np.nextafter.accumulate(np.concatenate([[start], np.full(4095, np.inf, np.float32)]
                                                     ).astype(np.float32))
        runs += [run, -run]
    v = np.concatenate(runs).astype(np.float32)
    v = v[np.abs(v) <= amax]
    q, s = _gpu_quantize(torch.from_numpy(v).cuda())
    ref_q, ref_s = Q.quantize(v)
    assert s == ref_s
    assert np.array_equal(q, ref_q), int(np.sum(q != ref_q))


def test_quantize_ties_round_to_even():
    # amax = 448 gives scale 1, so every value is its own quotient: all e4m3 midpoints
    grid = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (grid[:-1] + grid[1:]) / 2
    v = np.concatenate([[448.0], mids, -mids]).astype(np.float32)
    q, s = _gpu_quantize(torch.from_numpy(v).cuda())
    assert s == np.float32(1.0)
    assert np.array_equal(q, Q.quantize(v)[0])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_large_layer_size_sampled(dtype):
    shape = synth.CONFIGS[4]
    n = shape.N * shape.C * shape.D * shape.H * shape.W
    v = _values("normal", n, seed=4).to(dtype)
    q, s = _gpu_quantize(v.cuda())
    vf = v.float().numpy()
    ref_s = Q.scale_of(np.max(np.abs(vf)))
    assert s == ref_s
    idx = np.random.default_rng(0).integers(0, n, 200000)
    idx[:2] = [0, n - 1]
    assert np.array_equal(q[idx], Q.quantize_points(vf, idx, ref_s))


def _fused_inputs(cfg, dtype):
    shape = synth.CONFIGS[cfg]
    base = synth.make_config_inputs(cfg)        # e4m3 weights and their scale
    g = torch.Generator().manual_seed(500 + cfg)
    x = torch.randn((shape.N, shape.C, shape.D, shape.H, shape.W), generator=g).to(dtype)
    return shape, x, base["w"], base["sw"]


def _fused_run(shape, x, w, sw, **opts):
    s = shape
    plan = capi.conv3d_fp8_plan(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S, s.stride, s.pad,
                                **opts)
    info = capi.conv3d_fp8_get_info(plan)
    try:
        y = torch.full((s.N, s.K, info["Do"], info["Ho"], info["Wo"]), float("nan"),
                       dtype=torch.bfloat16, device="cuda")
        sx = torch.full((1,), float("nan"), device="cuda")
        swd = torch.tensor([sw], dtype=torch.float32, device="cuda")
        capi.conv3d_fp8_run_quantize_x(plan, x.cuda(), w.cuda(), swd, y, s.stride, s.pad, sx)
        torch.cuda.synchronize()
        assert capi.conv3d_fp8_check(plan) == capi.CONV3D_OK
        return y, np.float32(sx.item()), info
    finally:
        capi.conv3d_fp8_destroy(plan)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("route", [0, 1, 2, 4])
@pytest.mark.parametrize("cfg", [0, 1, 3])
def test_fused_run_full_output(cfg, route, dtype):
    shape, x, w, sw = _fused_inputs(cfg, dtype)
    y, sx, info = _fused_run(shape, x, w, sw, route=route)
    xq, ref_sx = Q.quantize(x.float().numpy())
    assert sx == ref_sx
    y64, yb = oracle.conv3d_fp8(xq.reshape(x.shape), w.numpy(), ref_sx, sw, shape.stride,
                                shape.pad)
    check_against(bits(y), y64, yb, f"fused quantise cfg {cfg} route {info['route']}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("cfg", [2, 4])
def test_fused_run_sampled_outputs(cfg, dtype):
    shape, x, w, sw = _fused_inputs(cfg, dtype)
    y, sx, info = _fused_run(shape, x, w, sw)
    assert not torch.isnan(y).any().item()
    xq, ref_sx = Q.quantize(x.float().numpy())
    assert sx == ref_sx
    idx = sample_indices(y.shape, 30000, seed=cfg)
    y64, yb = oracle.conv3d_fp8_points(xq.reshape(x.shape), w.numpy(), ref_sx, sw, idx,
                                       shape.stride, shape.pad)
    check_against(bits(y).ravel()[idx], y64, yb, f"fused quantise cfg {cfg}")


def test_fused_run_rejections():
    shape, x, w, sw = _fused_inputs(0, torch.float32)
    s = shape
    xd, wd = x.cuda(), w.cuda()
    swd = torch.tensor([sw], dtype=torch.float32, device="cuda")
    y = torch.full((1, s.K, 4, 8, 9), float("nan"), dtype=torch.bfloat16, device="cuda")
    cl = capi.conv3d_fp8_plan(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S, s.stride, s.pad,
                              input_layout=1)
    bf = capi.conv3d_bf16_plan(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S, s.stride, s.pad)
    ok = capi.conv3d_fp8_plan(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S, s.stride, s.pad)
    try:
        for plan in (cl, bf):
            assert capi.conv3d_fp8_run_quantize_x_status(plan, xd, wd, swd, y, s.stride,
                                                         s.pad) == capi.CONV3D_EINVAL
        assert capi.conv3d_fp8_run_quantize_x_status(ok, xd.view(-1)[1:], wd, swd, y, s.stride,
                                                     s.pad) == capi.CONV3D_EINVAL  # misaligned
        torch.cuda.synchronize()
        assert torch.isnan(y).all().item()
    finally:
        for plan in (cl, bf, ok):
            capi.conv3d_fp8_destroy(plan)
