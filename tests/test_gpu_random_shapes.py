"""Seeded random shapes, CUDA path vs the CPU oracle in full.

Each case draws a small 3D convolution (batch, channel multiples of 16, any K, filter sizes 1-3
per axis including even ones, pad 0-2 per axis, unit stride in every other case and strides 1-2
per axis otherwise, channel counts that are multiples of 32 in two cases of three, volumes from
one voxel to 20 x 20 x 20), runs
the library's own plan and one forced kernel (route x CTA pair, the first one the planner accepts
in a rotating order), and compares every output with the oracle under the shared gates. The
shapes are fixed by the seed, so a failure reproduces.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_implicit_gemm_gb300 import capi, synth
from _gpu_common import GpuConv, GpuConvBf16, bits, check_against, FROB_TOL_BF16, FROB64_TOL_BF16

pytestmark = pytest.mark.gpu

KERNELS = [dict(route=1, cta_pair=1), dict(route=2, cta_pair=1), dict(route=2, cta_pair=2),
           dict(route=3, cta_pair=2), dict(route=4, cta_pair=1)]
MAX_MACS = 1.5e8  # keeps the oracle to a fraction of a second a case


def random_shape(rng: np.random.Generator, unit_stride: bool, c32: bool) -> synth.ConvShape:
    while True:
        N = int(rng.integers(1, 4))
        C = 32 * int(rng.integers(1, 6)) if c32 else 16 * int(rng.integers(1, 11))
        K = int(rng.integers(1, 201))
        f = [int(v) for v in rng.integers(1, 4, size=3)]
        st = (1, 1, 1) if unit_stride else tuple(int(v) for v in rng.integers(1, 3, size=3))
        pd = tuple(int(rng.integers(0, min(2, f[i] - 1) + 1)) for i in range(3))
        dims = [int(v) for v in rng.integers(1, 21, size=3)]
        out = [(dims[i] + 2 * pd[i] - f[i]) // st[i] + 1 for i in range(3)]
        if min(out) < 1:
            continue
        macs = N * out[0] * out[1] * out[2] * K * C * f[0] * f[1] * f[2]
        if macs > MAX_MACS:
            continue
        return synth.ConvShape(N, C, dims[0], dims[1], dims[2], K, T=f[0], R=f[1], S=f[2],
                               stride=st, pad=pd)


def _shapes(count: int, seed: int):
    rng = np.random.default_rng(seed)
    return [random_shape(rng, unit_stride=(k % 2 == 0), c32=(k % 3 != 2)) for k in range(count)]


SHAPES = _shapes(64, 2024)


def _forced(shape, i: int, describe):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for j in range(len(KERNELS)):
        opts = KERNELS[(i + j) % len(KERNELS)]
        if describe(shape.N, shape.C, shape.D, shape.H, shape.W, shape.K, shape.T, shape.R,
                    shape.S, shape.stride, shape.pad, sms, **opts) == capi.CONV3D_OK:
            return opts
    return None


@pytest.mark.parametrize("i", range(len(SHAPES)))
def test_random_shape_e4m3(i):
    shape = SHAPES[i]
    inp = synth.make_inputs(shape, 500 + i)
    y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                shape.stride, shape.pad)
    forced = _forced(shape, i, capi.conv3d_fp8_describe_status)
    for opts in [{}] + ([forced] if forced else []):
        g = GpuConv(shape, inp, **opts)
        try:
            out = bits(g.run())
            res = check_against(out, y64, yb, f"{shape} {opts}")
            for k, v in opts.items():
                assert g.info[k] == v, (k, g.info[k], v)
            print(shape, opts, res, g.info["route"], g.info["splits"])
        finally:
            g.close()


@pytest.mark.parametrize("i", range(0, len(SHAPES), 3))
def test_random_shape_bf16(i):
    shape = SHAPES[i]
    inp = synth.make_inputs_bf16(shape, 900 + i)
    y64, yb = oracle.conv3d_bf16(synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["w"]),
                                 shape.stride, shape.pad)
    g = GpuConvBf16(shape, inp)
    try:
        out = bits(g.run())
        print(shape, check_against(out, y64, yb, str(shape), frob_tol=FROB_TOL_BF16,
                                   frob64_tol=FROB64_TOL_BF16))
    finally:
        g.close()
