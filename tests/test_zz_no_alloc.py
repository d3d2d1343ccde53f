"""The allocation-free entry point against the planned one and against the oracle.

conv3d_fp8_run_noalloc is for callers that cannot call cudaMalloc (a framework whose caching
allocator owns the device memory, a plugin interface with no way to request memory, a loop that
cannot take cudaFree's synchronisation). It keeps its scratch in one fixed device array that
every call reuses, so the test makes several calls in a row on different workloads, each one
finding the previous call's packed operands and partials still in the array:

  1. a stride-2 layer on the TMA im2col route, whose channels-last copy of x (no halo) fills the
     first megabyte of the array with nonzero bytes;
  2. a two-image layer on the padded-grid route packed by the tiled transpose (W % 4 == 0, 64
     channels): its packed copy of x carries a zero halo, and that halo now lies on the bytes
     call 1 left behind, so the transpose's blocks must rewrite it after their tiles;
  3. the two-image layer of the workloads (W = 15) on the padded-grid route, packed by items, whose
     halo lies on call 2's bytes;
  4. a 48-channel layer on the cp.async gather route, whose packed copy also has a halo;
  5. the deep stride-2 layer on the direct route (the explicit im2col of x in the array, split-K
     partials after it);
  6. the padded-row layer of the subject page (TMA im2col route, row guard on).

Each result must be bit for bit the planned run's (same kernels, same plan) and within the parity
gates against the oracle. A problem too big for the array is refused before anything runs.

This file sorts last so that a run stopping at its first failure has run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_implicit_gemm_gb300 import capi, synth
from _gpu_common import GpuConv, bits, check_against

pytestmark = pytest.mark.gpu

GATHER_48 = synth.ConvShape(2, 48, 4, 6, 5, 80, name="gather_2x48x4x6x5_k80_s1")
IM2COL_S2 = synth.ConvShape(1, 64, 16, 32, 32, 64, stride=2, name="im2col_1x64x16x32x32_k64_s2")
GRID_W16 = synth.ConvShape(2, 64, 8, 16, 16, 128, name="grid_2x64x8x16x16_k128_s1")


def _noalloc(g: GpuConv) -> np.ndarray:
    s = g.shape
    y = g.new_y()
    capi.conv3d_fp8_run_noalloc(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S, s.stride, s.pad,
                                g.x, g.w, g.sx, g.sw, y)
    torch.cuda.synchronize()
    return bits(y)


def _planned(g: GpuConv) -> np.ndarray:
    out = bits(g.run())
    assert capi.conv3d_fp8_check(g.plan) == capi.CONV3D_OK
    return out


def test_noalloc_matches_planned_run_and_oracle_on_calls_in_a_row():
    shapes = [(IM2COL_S2, synth.make_inputs(IM2COL_S2, 6464), 2),
              (GRID_W16, synth.make_inputs(GRID_W16, 1616), 3),
              (synth.CONFIGS[1], synth.make_config_inputs(1), 3),
              (GATHER_48, synth.make_inputs(GATHER_48, 4848), 1),
              (synth.CONFIGS[3], synth.make_config_inputs(3), 4),
              (synth.CONFIGS[0], synth.make_config_inputs(0), 2)]
    cases = []
    try:
        for shape, inp, route in shapes:
            g = GpuConv(shape, inp)
            cases.append((shape, inp, g))
            assert g.info["route"] == route, (shape.name, g.info["route"])
        planned = [_planned(g) for _, _, g in cases]
        got = []
        for _, _, g in cases:
            got.append(_noalloc(g))
            assert capi.conv3d_fp8_noalloc_check() == capi.CONV3D_OK
        for (shape, inp, g), ref, out in zip(cases, planned, got):
            assert np.array_equal(out, ref), (
                f"{shape.name}: {int(np.sum(out != ref))} outputs differ from the planned run")
            y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"],
                                        inp["sw"], shape.stride, shape.pad)
            check_against(out, y64, yb, f"no-alloc, {shape.name}")
    finally:
        for _, _, g in cases:
            g.close()


def test_noalloc_rejects_problems_beyond_its_scratch():
    s = synth.CONFIGS[4]  # packed operands alone need about 74 MB
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    scale = torch.ones(1, dtype=torch.float32, device="cuda")
    st = capi.conv3d_fp8_run_noalloc_status(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S,
                                            s.stride, s.pad, dummy, dummy, scale, scale, dummy)
    assert st == capi.CONV3D_EUNSUPPORTED
