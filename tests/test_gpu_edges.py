"""Degenerate and boundary shapes against the CPU oracle, in full, on every kernel that takes them:
one output channel, K not a multiple of the N tile, D = 1 (a 2D convolution), a filter as large as
the input (one output position per image), a stride larger than the filter, many tiny images, deep
C with few output channels, wide pads, filters of 729 and 1331 taps (the weight re-layout by
shared-memory tiles and its per-thread fallback)."""
import pytest
import torch

import oracle
from fp8_implicit_gemm_gb300 import capi, synth
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
    # 729 taps: one 16-byte weight chunk of every tap per tile (11.7 KB of the 16 KB tile)
    synth.ConvShape(1, 32, 9, 10, 11, 24, T=9, R=9, S=9, pad=2),
    # 1331 taps: a chunk of every tap exceeds the tile; the weights take the per-thread items
    synth.ConvShape(1, 16, 11, 11, 11, 16, T=11, R=11, S=11, pad=1),
    synth.ConvShape(1, 32, 11, 12, 11, 24, T=11, R=11, S=11, pad=(2, 1, 3)),
]
KERNELS = {"auto": {}, "gather-1cta": dict(route=1, cta_pair=1),
           "im2col-1cta": dict(route=2, cta_pair=1), "im2col-pair": dict(route=2, cta_pair=2),
           "grid-pair": dict(route=3, cta_pair=2), "direct-1cta": dict(route=4, cta_pair=1)}


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("i", range(len(EDGES)))
def test_edge_shape(i, kernel):
    shape = EDGES[i]
    opts = KERNELS[kernel]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if capi.conv3d_fp8_describe_status(shape.N, shape.C, shape.D, shape.H, shape.W, shape.K,
                                       shape.T, shape.R, shape.S, shape.stride, shape.pad, sms,
                                       **opts) != capi.CONV3D_OK:
        pytest.skip("the planner does not offer this kernel for this shape")
    inp = synth.make_inputs(shape, 900 + i)
    y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                shape.stride, shape.pad)
    g = GpuConv(shape, inp, **opts)
    try:
        check_against(bits(g.run()), y64, yb, f"{shape} {kernel}")
    finally:
        g.close()
