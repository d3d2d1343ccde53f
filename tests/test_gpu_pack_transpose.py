"""The tiled transpose of the operand pack (pack_x_transpose_kernel) at its edges, against the
oracle over the whole output.

That kernel copies an NCDHW x of e4m3 bytes or of the BF16 twin's bfloat16 elements (W % 4 == 0,
D*H*W*element-bytes % 16 == 0, C % 64 == 0) into the channels-last copy through a ring of 16 KB
tiles. The shapes below reach each of its forms: 64-channel groups (C = 64, 192) and 128-channel
groups, a W of 4 (a position group is a whole row), a last tile that holds one 16-byte run of its
channel planes, several images, padding 2 and stride 2, on the three routes that read the copy
(the cp.async gather and the padded grid, whose copies carry a zero halo, and TMA im2col, whose
copy has none). A wrong byte anywhere in the copy moves some output.
"""
import pytest

import oracle
from fp8_implicit_gemm_gb300 import synth
from _gpu_common import (FROB64_TOL_BF16, FROB_TOL_BF16, GpuConv, GpuConvBf16, bits,
                         check_against)

pytestmark = pytest.mark.gpu

SHAPES = [
    synth.ConvShape(2, 64, 4, 4, 4, 48),                 # 64-ch groups, 256-position tiles, 64 valid
    synth.ConvShape(1, 192, 3, 6, 8, 64),                # three 64-channel groups
    synth.ConvShape(3, 128, 5, 8, 20, 80),               # 128-ch groups, 800 = 6 x 128 + 32
    synth.ConvShape(1, 64, 4, 8, 16, 32, pad=2),         # halo of 2
    synth.ConvShape(2, 128, 6, 8, 16, 64, stride=2),     # stride 2 (gather and im2col routes)
    synth.ConvShape(1, 256, 1, 2, 8, 64),                # one 16-position run per channel plane
]
ROUTES = {"gather": dict(route=1, cta_pair=1), "im2col": dict(route=2, cta_pair=1),
          "grid": dict(route=3, cta_pair=2)}


def _cases():
    for i, s in enumerate(SHAPES):
        for name in ROUTES:
            if name == "grid" and s.stride != (1, 1, 1):
                continue  # the padded-grid route needs stride 1
            yield i, name


@pytest.mark.parametrize("i,route", list(_cases()))
def test_e4m3_transpose_edges(i, route):
    s = SHAPES[i]
    assert s.W % 4 == 0 and (s.D * s.H * s.W) % 16 == 0 and s.C % 64 == 0
    inp = synth.make_inputs(s, 4100 + i)
    y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                s.stride, s.pad)
    g = GpuConv(s, inp, **ROUTES[route])
    try:
        assert g.info["route"] == ROUTES[route]["route"]
        check_against(bits(g.run()), y64, yb, f"{s} {route}")
    finally:
        g.close()


@pytest.mark.parametrize("i,route", list(_cases()))
def test_bf16_transpose_edges(i, route):
    s = SHAPES[i]
    inp = synth.make_inputs_bf16(s, 4200 + i)
    y64, yb = oracle.conv3d_bf16(synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["w"]), s.stride,
                                 s.pad)
    g = GpuConvBf16(s, inp, **ROUTES[route])
    try:
        assert g.info["route"] == ROUTES[route]["route"]
        check_against(bits(g.run()), y64, yb, f"{s} {route} bf16", frob_tol=FROB_TOL_BF16,
                      frob64_tol=FROB64_TOL_BF16)
    finally:
        g.close()
