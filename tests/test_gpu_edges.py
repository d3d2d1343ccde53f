"""Degenerate and boundary shapes against the CPU oracle, in full, on every kernel that takes them:
one output channel, K not a multiple of the N tile, D = 1 (a 2D convolution), a filter as large as
the input (one output position per image), a stride larger than the filter, many tiny images, deep
C with few output channels, wide pads."""
import pytest

import oracle
from fp8_implicit_gemm_gb300 import synth
from _gpu_common import GpuConv, bits, check_against

pytestmark = pytest.mark.gpu

EDGES = [
    synth.ConvShape(1, 32, 4, 6, 8, 1),                                  # K = 1
    synth.ConvShape(2, 32, 3, 5, 6, 17),                                 # K = 17
    synth.ConvShape(1, 64, 2, 9, 10, 300),                               # 2 N tiles, the 2nd partial
    synth.ConvShape(2, 32, 1, 12, 14, 64, T=1, R=3, S=3, pad=(0, 1, 1)),  # D = 1
    synth.ConvShape(3, 32, 3, 3, 3, 48, pad=0),                          # filter = input: 1 output
    synth.ConvShape(2, 32, 7, 8, 9, 32, T=1, R=1, S=1, pad=0, stride=3),  # stride > filter
    synth.ConvShape(64, 32, 2, 2, 2, 32),                                # many tiny images
    synth.ConvShape(1, 1024, 2, 4, 4, 64),                               # deep C, few outputs
    synth.ConvShape(1, 32, 4, 5, 6, 32, pad=3, stride=(1, 2, 1)),        # pad 3, mixed stride
    synth.ConvShape(1, 32, 5, 4, 3, 40, T=3, R=1, S=3, pad=(1, 0, 1)),   # asymmetric filter
]
KERNELS = {"auto": {}, "gather-1cta": dict(route=1, cta_pair=1),
           "im2col-1cta": dict(route=2, cta_pair=1), "im2col-pair": dict(route=2, cta_pair=2),
           "grid-pair": dict(route=3, cta_pair=2)}


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("i", range(len(EDGES)))
def test_edge_shape(i, kernel):
    shape = EDGES[i]
    opts = KERNELS[kernel]
    if kernel == "grid-pair" and shape.stride != (1, 1, 1):
        pytest.skip("the padded-grid route needs stride 1")
    if kernel in ("im2col-1cta", "im2col-pair") and any(p > 15 for p in shape.pad):
        pytest.skip("im2col corners")
    inp = synth.make_inputs(shape, 900 + i)
    y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                shape.stride, shape.pad)
    g = GpuConv(shape, inp, **opts)
    try:
        check_against(bits(g.run()), y64, yb, f"{shape} {kernel}")
    finally:
        g.close()
