"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Every workload is compared in full, the two large ones (65536 and 244800 output positions, 8.4 M
and 62.7 M outputs) included, in the same launch configuration the benchmark times: the
whole-tensor Frobenius gate is the one the verification of the subject page applies to its worst
case ("Verification": the worst rel_err over the whole output). Every y is pre-filled with NaN,
so an element that is never written fails.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_implicit_gemm_gb300 import synth
from _gpu_common import GpuConv, bits, check_against, sample_indices

pytestmark = pytest.mark.gpu


def _full_case(shape, seed, **opts):
    inp = synth.make_inputs(shape, seed)
    y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                shape.stride, shape.pad)
    g = GpuConv(shape, inp, **opts)
    try:
        out = bits(g.run())
        assert out.shape == y64.shape
        return check_against(out, y64, yb, shape.name or str(shape)), g.info
    finally:
        g.close()


ROUTES = {"gather": 1, "im2col": 2, "grid": 3}
# (route, kernel): the cp.async gather route runs on one CTA, im2col on one CTA or on CTA pairs,
# the padded-grid route on CTA pairs
KERNELS = {"gather-1cta": dict(route=1, cta_pair=1), "im2col-1cta": dict(route=2, cta_pair=1),
           "im2col-pair": dict(route=2, cta_pair=2), "grid-pair": dict(route=3, cta_pair=2),
           "direct-1cta": dict(route=4, cta_pair=1)}


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("cfg", [0, 1, 3])
def test_config_full_output(cfg, kernel):
    if kernel == "grid-pair" and cfg == 3:
        pytest.skip("the padded-grid route needs stride 1")
    res, info = _full_case(synth.CONFIGS[cfg], synth.config_seed(cfg), **KERNELS[kernel])
    assert info["route"] == KERNELS[kernel]["route"]
    assert info["cta_pair"] == KERNELS[kernel]["cta_pair"]
    print(cfg, kernel, res, info["splits"], info["block_n"])


# The oracle's full output of one large workload at a time (config 4: 62.7 M outputs, about 45 s on
# 16 host cores and 0.6 GB), shared by the kernel variants of that workload.
_LARGE = {}


def _large_reference(cfg):
    if cfg not in _LARGE:
        _LARGE.clear()
        shape = synth.CONFIGS[cfg]
        inp = synth.make_config_inputs(cfg)
        y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                    shape.stride, shape.pad)
        _LARGE[cfg] = (inp, y64, yb)
    return _LARGE[cfg]


@pytest.mark.parametrize("cfg,kernel", [(c, k) for c in (2, 4)
                                        for k in ("auto", "im2col-1cta", "im2col-pair")] +
                         [(2, "direct-1cta")])
def test_config_full_output_large(cfg, kernel):
    shape = synth.CONFIGS[cfg]
    inp, y64, yb = _large_reference(cfg)
    g = GpuConv(shape, inp, **KERNELS.get(kernel, {}))
    try:
        out = bits(g.run())
        assert out.shape == y64.shape
        res = check_against(out, y64, yb, f"{shape.name} [{kernel}]")
        print(f"full-output parity: config {cfg} [{kernel}] plan route {g.info['route']} "
              f"pair {g.info['cta_pair']}: frobenius {res['frob']:.4e}, bf16 flips "
              f"{res['bf16_flips']} of {res['n']} ({res['bf16_flips'] / res['n']:.3e})")
        # the oracle's points mode on the structured edge indices (first and last rows of every
        # image, the padded-tile edge, the volume's faces) agrees with its full mode bit for bit
        idx = sample_indices(g.out_shape, 2000, seed=cfg)
        p64, pb = oracle.conv3d_fp8_points(inp["x"].numpy(), inp["w"].numpy(), inp["sx"],
                                           inp["sw"], idx, shape.stride, shape.pad)
        assert np.array_equal(pb, yb.ravel()[idx]) and np.array_equal(p64, y64.ravel()[idx])
    finally:
        g.close()


# Odd shapes: channel counts that are multiples of 16 but not 32 (K_gemm tail of 16 bytes), K not a
# multiple of the N tile, W = 1, stride 2 on odd sizes, n > 1 tiles that straddle images,
# 1x1x1 and 1x3x3 filters, pad 0 and 2, anisotropic stride/pad, tiny volumes.
ODD = [
    synth.ConvShape(1, 16, 3, 5, 7, 16),
    synth.ConvShape(2, 48, 4, 6, 5, 80),
    synth.ConvShape(3, 32, 5, 7, 9, 100, stride=2),
    synth.ConvShape(1, 64, 6, 9, 1, 32, T=3, R=3, S=1, pad=(1, 1, 0)),
    synth.ConvShape(2, 16, 4, 4, 4, 48, T=1, R=1, S=1, pad=0),
    synth.ConvShape(1, 32, 2, 11, 13, 64, T=1, R=3, S=3, pad=(0, 1, 1)),
    synth.ConvShape(1, 16, 7, 7, 7, 16, pad=2),
    synth.ConvShape(1, 32, 9, 10, 11, 96, stride=(1, 2, 3), pad=(0, 1, 2)),
    synth.ConvShape(1, 16, 1, 1, 1, 16, pad=1),
    synth.ConvShape(2, 128, 3, 17, 19, 256),
    synth.ConvShape(1, 272, 2, 5, 6, 40),
]


@pytest.mark.parametrize("i", range(len(ODD)))
def test_odd_shapes(i):
    res, info = _full_case(ODD[i], 77 + i)
    print(ODD[i], res, info["splits"], info["block_n"], info["route"])


@pytest.mark.parametrize("i", [i for i, s in enumerate(ODD) if s.C % 32 == 0])
def test_odd_shapes_gather_route(i):
    res, info = _full_case(ODD[i], 77 + i, route=ROUTES["gather"])
    assert info["route"] == ROUTES["gather"]


@pytest.mark.parametrize("i", [i for i, s in enumerate(ODD)
                               if s.C % 32 == 0 and s.stride == (1, 1, 1)])
def test_odd_shapes_grid_route(i):
    res, info = _full_case(ODD[i], 77 + i, route=3)
    assert info["route"] == 3


@pytest.mark.parametrize("i", range(len(ODD)))
def test_odd_shapes_direct_route(i):
    res, info = _full_case(ODD[i], 77 + i, route=4)
    assert info["route"] == 4 and info["cta_pair"] == 1


@pytest.mark.parametrize("i", [i for i, s in enumerate(ODD) if s.C % 32 == 0])
def test_odd_shapes_one_cta(i):
    res, info = _full_case(ODD[i], 77 + i, cta_pair=1)
    assert info["cta_pair"] == 1


@pytest.mark.parametrize("kernel", ["im2col-1cta", "im2col-pair", "grid-pair"])
@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_forced_splits_config1(splits, kernel):
    res, info = _full_case(synth.CONFIGS[1], synth.config_seed(1), splits=splits, **KERNELS[kernel])
    # a split count is normalised so that no split is empty: ceil(kb / ceil(kb / requested));
    # the grid route has 9 K groups on this layer, the others 14 K blocks
    kb = info["k_blocks"]
    per = -(-kb // min(splits, kb))
    assert info["splits"] == -(-kb // per)


@pytest.mark.parametrize("kernel", ["im2col-1cta", "im2col-pair", "grid-pair"])
@pytest.mark.parametrize("block_n", [32, 64, 128, 256])
def test_forced_block_n(block_n, kernel):
    shape = synth.ConvShape(2, 32, 4, 6, 10, 200)
    res, info = _full_case(shape, 5, block_n=block_n, **KERNELS[kernel])
    assert info["block_n"] == block_n


@pytest.mark.parametrize("kernel", ["im2col-1cta", "im2col-pair", "grid-pair"])
def test_max_ctas_small_grid_many_tiles(kernel):
    # 2 CTAs (one pair) walk all tiles: exercises the TMEM double buffer and stage-ring wrap-around
    res, info = _full_case(synth.CONFIGS[1], synth.config_seed(1), max_ctas=2, splits=1,
                           **KERNELS[kernel])
    assert info["grid"] == 2


# A CTA cap that leaves a mostly idle last wave: its tiles are split along K over the idle slots
# while the others are computed whole, in one launch (whole tiles store bf16, split tiles fp32
# partials that the reduction then sums).
# A CTA cap leaves a last wave at most half full; the tiles' K loops (54 or 18 K blocks of N = 256
# MMAs) are long enough for the planner to split that wave's tiles along K.
TAIL_SHAPE = synth.ConvShape(1, 256, 8, 10, 12, 256)
TAIL_CASES = {"gather-1cta": 6, "im2col-1cta": 6, "im2col-pair": 6, "grid-pair": 8}


@pytest.mark.parametrize("kernel", list(TAIL_CASES))
def test_tail_tiles_split_along_k(kernel):
    res, info = _full_case(TAIL_SHAPE, 2718, max_ctas=TAIL_CASES[kernel], **KERNELS[kernel])
    tiles = info["m_tiles"] * info["n_tiles"]
    assert 0 < info["full_tiles"] < tiles and info["splits"] > 1, info


# Channels-last input (input_layout = 1): the TMA routes read the caller's NDHWC x directly (the
# padded-grid route through an im2col traversal of its zero-padded grid), the gather route copies
# it into its zero-padded buffer.
@pytest.mark.parametrize("kernel", [k for k in KERNELS if k != "direct-1cta"])
@pytest.mark.parametrize("cfg", [0, 1, 3])
def test_channels_last_input_full_output(cfg, kernel):
    if kernel == "grid-pair" and cfg == 3:
        pytest.skip("the padded-grid route needs stride 1")
    res, info = _full_case(synth.CONFIGS[cfg], synth.config_seed(cfg), input_layout=1,
                           **KERNELS[kernel])
    assert info["route"] == KERNELS[kernel]["route"]


@pytest.mark.parametrize("cfg", [2, 4])
def test_channels_last_input_sampled_outputs(cfg):
    shape = synth.CONFIGS[cfg]
    inp = synth.make_config_inputs(cfg)
    g = GpuConv(shape, inp, input_layout=1)
    try:
        y = g.run()
        assert not torch.isnan(y).any().item(), "some outputs never written"
        idx = sample_indices(g.out_shape, 60000, seed=50 + cfg)
        y64, yb = oracle.conv3d_fp8_points(inp["x"].numpy(), inp["w"].numpy(), inp["sx"],
                                           inp["sw"], idx, shape.stride, shape.pad)
        print(cfg, check_against(bits(y).ravel()[idx], y64, yb, shape.name))
    finally:
        g.close()


@pytest.mark.parametrize("i", range(len(ODD)))
def test_channels_last_input_odd_shapes(i):
    res, info = _full_case(ODD[i], 77 + i, input_layout=1)
    print(ODD[i], res, info["route"])


@pytest.mark.parametrize("i", [i for i, s in enumerate(ODD)
                               if s.C % 32 == 0 and s.stride == (1, 1, 1)])
def test_channels_last_input_odd_shapes_grid_route(i):
    res, info = _full_case(ODD[i], 77 + i, input_layout=1, route=3)
    assert info["route"] == 3


def test_split_k_is_reproducible_and_close_across_split_counts():
    shape = synth.CONFIGS[3]
    inp = synth.make_config_inputs(3)
    outs = {}
    for splits, pair in ((1, 1), (4, 1), (27, 1), (27, 2)):
        g = GpuConv(shape, inp, splits=splits, cta_pair=pair)
        try:
            a = bits(g.run())
            b = bits(g.run())
            assert np.array_equal(a, b), f"splits={splits} not bitwise reproducible"
            outs[(splits, pair)] = a
        finally:
            g.close()
    y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                shape.stride, shape.pad)
    for s, a in outs.items():
        check_against(a, y64, yb, f"splits={s}")


def test_plans_with_different_tiles_coexist():
    """A plan created after another one (with a different shared-memory footprint) must not break
    the first one's launches."""
    s0 = synth.CONFIGS[0]
    inp = synth.make_config_inputs(0)
    big = GpuConv(s0, inp, block_n=96, splits=1, cta_pair=1)   # 7 stages of 28 KB
    small = GpuConv(s0, inp, block_n=32, splits=1, cta_pair=2)  # pairs, 8 stages of 18 KB
    try:
        y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                    s0.stride, s0.pad)
        check_against(bits(big.run()), y64, yb, "first plan after a second was created")
        check_against(bits(small.run()), y64, yb, "second plan")
    finally:
        big.close()
        small.close()
