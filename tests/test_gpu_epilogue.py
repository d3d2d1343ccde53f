"""The hardware-bounded (TMA-store) epilogue, option epilogue = 2, against the CPU oracle.

Whole tiles leave through TMA stores of a tensor map of y viewed as [N][K][dhw]: rows past the
end of an image (the padded rows of the last tile among them) and columns past K are dropped by
the TMA unit, rows spilling into a later image take the explicit guarded stores. Every y starts
NaN-filled, so an element never written fails; the 200-repeat test is the subject page's
verification ("Verification": the padded-row race showed up in about 1 launch in 17) on its own
failing shape.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_implicit_gemm_gb300 import capi, synth
from _gpu_common import GpuConv, GpuConvBf16, NAN_BF16, bits, check_against

pytestmark = pytest.mark.gpu

KERNELS = {"gather-1cta": dict(route=1, cta_pair=1), "im2col-1cta": dict(route=2, cta_pair=1),
           "im2col-pair": dict(route=2, cta_pair=2)}


def _full(shape, seed, **opts):
    inp = synth.make_inputs(shape, seed)
    y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                shape.stride, shape.pad)
    g = GpuConv(shape, inp, epilogue=2, **opts)
    try:
        assert g.info["epilogue"] == 2
        out = bits(g.run())
        return check_against(out, y64, yb, str(shape)), g.info
    finally:
        g.close()


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("cfg", [0, 1, 3])
def test_config_full_output(cfg, kernel):
    _full(synth.CONFIGS[cfg], synth.config_seed(cfg), **KERNELS[kernel])


# dhw a multiple of 8; tiles that cross image boundaries (config 1 on pairs: 1920 = 7.5 * 256),
# several images per tile (dhw = 8 and 24), split tiles next to whole ones
SHAPES = [
    synth.ConvShape(40, 32, 2, 2, 2, 16),                      # dhw = 8: a tile spans 16 images
    synth.ConvShape(9, 48, 2, 3, 4, 40),                       # dhw = 24, K not a multiple of 32
    synth.ConvShape(2, 48, 4, 6, 5, 80),                       # dhw = 120
    synth.ConvShape(3, 32, 4, 4, 8, 96, T=1, R=3, S=3, pad=(0, 1, 1)),   # dhw = 128
    synth.ConvShape(2, 16, 4, 9, 10, 200, stride=(1, 1, 1), pad=(1, 1, 1)),  # 16 channels: gather
]


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("i", range(len(SHAPES)))
def test_image_crossing_tiles(i, kernel):
    shape = SHAPES[i]
    if shape.C % 32 != 0 and kernel != "gather-1cta":
        pytest.skip("16-byte channel rows take the gather route")
    _full(shape, 300 + i, **KERNELS[kernel])


@pytest.mark.parametrize("kernel", ["im2col-1cta", "im2col-pair"])
def test_whole_and_split_tiles_together(kernel):
    # a CTA cap leaves a last wave at most half full, and the K loops are long enough to split it
    res, info = _full(synth.ConvShape(1, 256, 8, 10, 12, 256), 2720, max_ctas=6, **KERNELS[kernel])
    assert 0 < info["full_tiles"] < info["m_tiles"] * info["n_tiles"]


def test_bf16_twin():
    shape = synth.CONFIGS[1]
    inp = synth.make_config_inputs_bf16(1)
    y64, yb = oracle.conv3d_bf16(synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["w"]),
                                 shape.stride, shape.pad)
    g = GpuConvBf16(shape, inp, epilogue=2, route=2)
    try:
        check_against(bits(g.run()), y64, yb, "bf16", frob_tol=1e-3, frob64_tol=2.0 ** -8)
    finally:
        g.close()


@pytest.mark.parametrize("kernel", ["im2col-1cta", "im2col-pair"])
def test_page_case_200_repeats(kernel):
    shape = synth.CONFIGS[0]  # 1x96x4x8x9 -> 96: npq = 288, the padded rows alias live outputs
    inp = synth.make_config_inputs(0)
    g = GpuConv(shape, inp, epilogue=2, **KERNELS[kernel])
    try:
        y = g.new_y()
        nan16 = np.int16(np.uint16(NAN_BF16).view(np.int16))
        first = None
        for rep in range(200):
            y.view(torch.int16).fill_(nan16)
            g.run(y)
            if first is None:
                first = y.clone()
            else:
                assert torch.equal(y.view(torch.int16), first.view(torch.int16)), rep
        y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                    shape.stride, shape.pad)
        check_against(bits(first), y64, yb, "200 repeats")
        assert capi.conv3d_fp8_check(g.plan) == capi.CONV3D_OK
    finally:
        g.close()


def test_bounded_wait_with_tma_epilogue():
    shape = synth.CONFIGS[0]
    inp = synth.make_config_inputs(0)
    for kernel in ("im2col-1cta", "im2col-pair"):
        bad = GpuConv(shape, inp, debug_flags=1, wait_timeout_ms=200, splits=1, epilogue=2,
                      **KERNELS[kernel])
        try:
            bad.run()
            assert capi.conv3d_fp8_check(bad.plan) == capi.CONV3D_EDEVICE
        finally:
            bad.close()
    _full(shape, synth.config_seed(0), route=2)
