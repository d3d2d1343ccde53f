"""A wider seeded sweep of shapes and plan options, CUDA path vs the CPU oracle in full.

Beyond the first sweep's ranges: filters of 1-5 taps per axis, pads 0-3 and strides 1-3 chosen
per axis independently (so pads may exceed half the filter and strides may skip input voxels),
channel counts 16-256, K 1-300, volumes up to 32 along an axis; half the shapes have unit stride.
Each shape runs the library's own plan and one plan with seeded random options (split count, CTA
cap, N tile, and a route / CTA-pair choice: the padded grid for half the shapes it applies to),
skipping an option set the planner refuses; a third of the shapes also run the bfloat16 twin with
the same options. Every output is compared with the oracle under the shared gates.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_implicit_gemm_gb300 import capi, synth
from _gpu_common import GpuConv, GpuConvBf16, bits, check_against, FROB_TOL_BF16, FROB64_TOL_BF16

pytestmark = pytest.mark.gpu

MAX_MACS = 2.0e8
KERNELS = [{}, dict(route=1, cta_pair=1), dict(route=2, cta_pair=1), dict(route=2, cta_pair=2),
           dict(route=3, cta_pair=2), dict(route=4, cta_pair=1)]


def wide_shape(rng: np.random.Generator) -> synth.ConvShape:
    while True:
        N = int(rng.integers(1, 4))
        C = 16 * int(rng.integers(1, 17))
        K = int(rng.integers(1, 301))
        f = [int(v) for v in rng.integers(1, 6, size=3)]
        st = tuple(int(v) for v in rng.integers(1, 4, size=3))
        if rng.random() < 0.5:  # half the shapes at unit stride: the padded-grid route's domain
            st = (1, 1, 1)
        pd = tuple(int(v) for v in rng.integers(0, 4, size=3))
        dims = [int(v) for v in rng.integers(1, 33, size=3)]
        out = [(dims[i] + 2 * pd[i] - f[i]) // st[i] + 1 for i in range(3)]
        if min(out) < 1:
            continue
        macs = N * out[0] * out[1] * out[2] * K * C * f[0] * f[1] * f[2]
        if macs > MAX_MACS:
            continue
        return synth.ConvShape(N, C, dims[0], dims[1], dims[2], K, T=f[0], R=f[1], S=f[2],
                               stride=st, pad=pd)


def wide_options(rng: np.random.Generator, shape: synth.ConvShape) -> dict:
    o = dict(KERNELS[int(rng.integers(0, len(KERNELS)))])
    if shape.stride == (1, 1, 1) and shape.C % 32 == 0 and rng.random() < 0.5:
        o = dict(route=3, cta_pair=2)
    o["splits"] = [0, 0, 2, 3, 5][int(rng.integers(0, 5))]
    o["max_ctas"] = [0, 0, 4, 10, 40][int(rng.integers(0, 5))]
    o["block_n"] = [0, 0, 32, 64, 128, 256][int(rng.integers(0, 6))]
    return o


def _cases(count: int, seed: int):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(count):
        shape = wide_shape(rng)
        cases.append((shape, wide_options(rng, shape)))
    return cases


CASES = _cases(48, 9090)


def _accepted(describe, shape, opts) -> bool:
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return describe(shape.N, shape.C, shape.D, shape.H, shape.W, shape.K, shape.T, shape.R,
                    shape.S, shape.stride, shape.pad, sms, **opts) == capi.CONV3D_OK


@pytest.mark.parametrize("i", range(len(CASES)))
def test_wide_random_shape_e4m3(i):
    shape, opts = CASES[i]
    inp = synth.make_inputs(shape, 900 + i)
    y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                shape.stride, shape.pad)
    variants = [{}]
    if _accepted(capi.conv3d_fp8_describe_status, shape, opts):
        variants.append(opts)
    for o in variants:
        g = GpuConv(shape, inp, **o)
        try:
            out = bits(g.run())
            check_against(out, y64, yb, f"{shape} {o}")
            assert capi.conv3d_fp8_check(g.plan) == capi.CONV3D_OK
        finally:
            g.close()


@pytest.mark.parametrize("i", [i for i in range(len(CASES)) if i % 3 == 0])
def test_wide_random_shape_bf16(i):
    shape, opts = CASES[i]
    inp = synth.make_inputs_bf16(shape, 950 + i)
    y64, yb = oracle.conv3d_bf16(synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["w"]),
                                 shape.stride, shape.pad)
    variants = [{}]
    if _accepted(capi.conv3d_bf16_describe_status, shape, opts):
        variants.append(opts)
    for o in variants:
        g = GpuConvBf16(shape, inp, **o)
        try:
            check_against(bits(g.run()), y64, yb, f"bf16 {shape} {o}", frob_tol=FROB_TOL_BF16,
                          frob64_tol=FROB64_TOL_BF16)
        finally:
            g.close()
