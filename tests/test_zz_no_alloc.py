"""The allocation-free entry point against the planned one.

conv3d_fp8_run_noalloc is for callers that cannot call cudaMalloc (a framework whose caching
allocator owns the device memory, a plugin interface with no way to request memory, a loop that
cannot take cudaFree's synchronisation). It keeps its scratch in one fixed device array that
every call reuses, so the test makes two calls in a row on different workloads -- the second one
finds the first one's packed operands and partials still in the array -- and checks each against
conv3d_fp8_run on a plan, within the parity tolerances of the other GPU tests. It also checks
that a problem too big for the array is refused before anything runs.

This file sorts last so that a run stopping at its first failure has run every other test.
"""
import numpy as np
import pytest
import torch

from fp8_implicit_gemm_gb300 import capi, synth
from _gpu_common import GpuConv, bits, check_against

pytestmark = pytest.mark.gpu


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


def test_noalloc_matches_planned_run_on_two_calls_in_a_row():
    # a split-K workload (partials in the array), then the padded-row one (row guard on): the
    # second call runs on an array still holding the first call's data
    cases = []
    for cfg in (3, 0):
        g = GpuConv(synth.CONFIGS[cfg], synth.make_config_inputs(cfg))
        cases.append((cfg, g, _planned(g)))
    try:
        outs = [_noalloc(g) for _, g, _ in cases]
        for (cfg, g, ref), got in zip(cases, outs):
            ref64 = (ref.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            check_against(got, ref64, ref, f"no-alloc vs planned, config {cfg}")
    finally:
        for _, g, _ in cases:
            g.close()


def test_noalloc_rejects_problems_beyond_its_scratch():
    s = synth.CONFIGS[4]  # packed operands alone need about 74 MB
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    scale = torch.ones(1, dtype=torch.float32, device="cuda")
    st = capi.conv3d_fp8_run_noalloc_status(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S,
                                            s.stride, s.pad, dummy, dummy, scale, scale, dummy)
    assert st == capi.CONV3D_EUNSUPPORTED
