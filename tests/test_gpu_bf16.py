"""The BF16-input twin (tcgen05.mma kind::f16) against its CPU oracle, through the C ABI.

The per-element gate of the e4m3 path (|d| <= 2^-7 |ref| + 1e-3 against the oracle's fp64 value)
and Frobenius gates derived for bfloat16 inputs (see _gpu_common.FROB_TOL_BF16), on the same
workloads with bfloat16 inputs
(x ~ N(0,1), w ~ N(0, 1/(C*T*R*S))): every route and kernel, odd shapes, forced split counts,
the split tail, channels-last input, NaN-prefilled repeats and the bounded-wait error path.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_implicit_gemm_gb300 import capi, synth
from _gpu_common import (FROB64_TOL_BF16, FROB_TOL_BF16, GpuConvBf16, NAN_BF16, bits,
                         check_against, sample_indices)


def check_bf16(gpu_bits, y64, yb, what):
    return check_against(gpu_bits, y64, yb, what, frob_tol=FROB_TOL_BF16,
                         frob64_tol=FROB64_TOL_BF16)

pytestmark = pytest.mark.gpu

KERNELS = {"gather-1cta": dict(route=1, cta_pair=1), "im2col-1cta": dict(route=2, cta_pair=1),
           "im2col-pair": dict(route=2, cta_pair=2), "grid-pair": dict(route=3, cta_pair=2),
           "direct-1cta": dict(route=4, cta_pair=1)}


def _oracle_full(shape, inp):
    return oracle.conv3d_bf16(synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["w"]),
                              shape.stride, shape.pad)


def _full_case(shape, seed, **opts):
    inp = synth.make_inputs_bf16(shape, seed)
    y64, yb = _oracle_full(shape, inp)
    g = GpuConvBf16(shape, inp, **opts)
    try:
        out = bits(g.run())
        assert out.shape == y64.shape
        return check_bf16(out, y64, yb, shape.name or str(shape)), g.info
    finally:
        g.close()


def _sampled_case(cfg, seed_off=0, **opts):
    shape = synth.CONFIGS[cfg]
    inp = synth.make_config_inputs_bf16(cfg)
    g = GpuConvBf16(shape, inp, **opts)
    try:
        y = g.run()
        assert not torch.isnan(y).any().item(), "some outputs never written"
        idx = sample_indices(g.out_shape, 40000, seed=cfg + seed_off)
        y64, yb = oracle.conv3d_bf16_points(synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["w"]),
                                            idx, shape.stride, shape.pad)
        return check_bf16(bits(y).ravel()[idx], y64, yb, shape.name), g.info
    finally:
        g.close()


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("cfg", [0, 1, 3])
def test_config_full_output(cfg, kernel):
    if kernel == "grid-pair" and cfg == 3:
        pytest.skip("the padded-grid route needs stride 1")
    res, info = _full_case(synth.CONFIGS[cfg], synth.config_seed(cfg), **KERNELS[kernel])
    assert info["route"] == KERNELS[kernel]["route"]
    assert info["cta_pair"] == KERNELS[kernel]["cta_pair"]


@pytest.mark.parametrize("cfg", [2, 4])
def test_config_sampled_outputs(cfg):
    res, info = _sampled_case(cfg)
    print(cfg, res, info["route"], info["splits"], info["full_tiles"])


@pytest.mark.parametrize("cfg", [2, 4])
def test_channels_last_input_sampled_outputs(cfg):
    res, info = _sampled_case(cfg, seed_off=7, input_layout=1)


ODD = [
    synth.ConvShape(1, 16, 3, 5, 7, 16),
    synth.ConvShape(2, 48, 4, 6, 5, 80),
    synth.ConvShape(3, 32, 5, 7, 9, 100, stride=2),
    synth.ConvShape(1, 64, 6, 9, 1, 32, T=3, R=3, S=1, pad=(1, 1, 0)),
    synth.ConvShape(2, 16, 4, 4, 4, 48, T=1, R=1, S=1, pad=0),
    synth.ConvShape(1, 32, 2, 11, 13, 64, T=1, R=3, S=3, pad=(0, 1, 1)),
    synth.ConvShape(1, 8, 7, 7, 7, 16, pad=2),                 # 16 bytes per pixel: gather
    synth.ConvShape(1, 24, 9, 10, 11, 96, stride=(1, 2, 3), pad=(0, 1, 2)),  # 48 bytes: gather
    synth.ConvShape(1, 16, 1, 1, 1, 16, pad=1),
    synth.ConvShape(2, 128, 3, 17, 19, 256),
    synth.ConvShape(1, 136, 2, 5, 6, 40),
    # 8-pixel pack items (W % 8 == 0): pixel group fastest below 16 chunks a pixel, chunk fastest
    # from there on
    synth.ConvShape(2, 32, 4, 6, 8, 64),
    synth.ConvShape(1, 64, 3, 5, 16, 48),
    synth.ConvShape(1, 128, 2, 4, 24, 64),
    synth.ConvShape(2, 256, 2, 3, 8, 32, stride=2),
]


@pytest.mark.parametrize("i", range(len(ODD)))
def test_odd_shapes(i):
    res, info = _full_case(ODD[i], 177 + i)
    print(ODD[i], res, info["route"], info["splits"])


@pytest.mark.parametrize("i", [i for i, s in enumerate(ODD) if s.C % 16 == 0])
def test_odd_shapes_channels_last_input(i):
    _full_case(ODD[i], 177 + i, input_layout=1)


@pytest.mark.parametrize("kernel", ["im2col-1cta", "im2col-pair", "grid-pair"])
@pytest.mark.parametrize("splits", [2, 5])
def test_forced_splits(splits, kernel):
    res, info = _full_case(synth.CONFIGS[1], synth.config_seed(1), splits=splits,
                           **KERNELS[kernel])
    assert info["splits"] > 1


@pytest.mark.parametrize("kernel", ["im2col-1cta", "grid-pair"])
def test_tail_tiles_split_along_k(kernel):
    # a CTA cap leaves a last wave at most half full, and the K loops are long enough to split it
    res, info = _full_case(synth.ConvShape(1, 256, 8, 10, 12, 256), 2719,
                           max_ctas={"im2col-1cta": 6, "grid-pair": 8}[kernel], **KERNELS[kernel])
    assert 0 < info["full_tiles"] < info["m_tiles"] * info["n_tiles"]


@pytest.mark.parametrize("cfg,repeats", [(0, 50), (4, 20)])
def test_repeated_launches_write_every_element_once(cfg, repeats):
    shape = synth.CONFIGS[cfg]
    inp = synth.make_config_inputs_bf16(cfg)
    g = GpuConvBf16(shape, inp)
    try:
        y = g.new_y()
        nan16 = np.int16(np.uint16(NAN_BF16).view(np.int16))
        first = None
        for rep in range(repeats):
            y.view(torch.int16).fill_(nan16)
            g.run(y)
            if first is None:
                first = y.clone()
                assert not torch.isnan(first).any().item()
            else:
                assert torch.equal(y.view(torch.int16), first.view(torch.int16)), rep
        assert capi.conv3d_fp8_check(g.plan) == capi.CONV3D_OK
    finally:
        g.close()


@pytest.mark.parametrize("kernel", [dict(cta_pair=1, route=2), dict(cta_pair=2, route=3),
                                    dict(cta_pair=1, route=4)])
def test_bounded_wait_reports_instead_of_hanging(kernel):
    shape = synth.CONFIGS[0]
    inp = synth.make_config_inputs_bf16(0)
    bad = GpuConvBf16(shape, inp, debug_flags=1, wait_timeout_ms=200, splits=1, **kernel)
    try:
        bad.run()
        assert capi.conv3d_fp8_check(bad.plan) == capi.CONV3D_EDEVICE
        assert capi.conv3d_fp8_check(bad.plan) == capi.CONV3D_OK
    finally:
        bad.close()
    _full_case(shape, synth.config_seed(0))


def test_plan_types_do_not_mix():
    shape = synth.CONFIGS[0]
    inp = synth.make_config_inputs_bf16(0)
    g = GpuConvBf16(shape, inp)
    try:
        y = g.new_y()
        one = torch.ones(1, device="cuda")
        assert capi.conv3d_fp8_run_status(g.plan, g.x, g.w, one, one, y, shape.stride,
                                          shape.pad) == capi.CONV3D_EINVAL
        fp8 = capi.conv3d_fp8_plan(shape.N, shape.C, shape.D, shape.H, shape.W, shape.K, shape.T,
                                   shape.R, shape.S, shape.stride, shape.pad)
        try:
            assert capi.conv3d_bf16_run_status(fp8, g.x, g.w, y, shape.stride,
                                               shape.pad) == capi.CONV3D_EINVAL
        finally:
            capi.conv3d_fp8_destroy(fp8)
        torch.cuda.synchronize()
        assert torch.isnan(y).all().item()
    finally:
        g.close()
