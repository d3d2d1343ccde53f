"""The host-buffer entry points, conv3d_fp8_run_host and conv3d_bf16_run_host, through the C ABI.

Each run copies x, w (and the e4m3 scales) from host memory into the plan's device buffers, runs
the same kernels as the device-pointer entry points and copies y back, all on one stream. So its
output must be bit for bit the device-pointer run's of the same plan and inputs, whichever host
memory the caller passes (page-locked or pageable), across consecutive calls that reuse the
plan's device buffers, and within the parity gates against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_implicit_gemm_gb300 import capi, synth
from _gpu_common import GpuConv, bits, check_against

pytestmark = pytest.mark.gpu


def _host(t: torch.Tensor, pinned: bool) -> torch.Tensor:
    t = t.contiguous().cpu()
    return t.pin_memory() if pinned else t.clone()


def _run_host(g: GpuConv, inp: dict, pinned: bool, layout: int = 0) -> np.ndarray:
    x = inp["x"]
    if layout == 1:
        x = x.permute(0, 2, 3, 4, 1)
    xh, wh = _host(x, pinned), _host(inp["w"], pinned)
    sh = _host(torch.tensor([inp["sx"], inp["sw"]], dtype=torch.float32), pinned)
    yh = _host(torch.full(g.out_shape, float("nan"), dtype=torch.bfloat16), pinned)
    stream = torch.cuda.Stream()
    capi.conv3d_fp8_run_host(g.plan, xh, wh, sh, yh, g.shape.stride, g.shape.pad, stream)
    stream.synchronize()
    assert capi.conv3d_fp8_check(g.plan) == capi.CONV3D_OK
    return bits(yh)


@pytest.mark.parametrize("cfg", [0, 1, 3])
@pytest.mark.parametrize("pinned", [True, False])
def test_run_host_matches_device_run_and_oracle(cfg, pinned):
    shape, inp = synth.CONFIGS[cfg], synth.make_config_inputs(cfg)
    g = GpuConv(shape, inp)
    try:
        ref = bits(g.run())
        torch.cuda.synchronize()
        out = _run_host(g, inp, pinned)
        assert np.array_equal(out, ref), f"{int(np.sum(out != ref))} outputs differ"
        y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                    shape.stride, shape.pad)
        check_against(out, y64, yb, f"run_host, {shape.name}")
    finally:
        g.close()


def test_run_host_consecutive_inputs_and_channels_last():
    # two input sets through one plan's device buffers, then a channels-last plan
    shape = synth.CONFIGS[1]
    sets = [synth.make_inputs(shape, 31), synth.make_inputs(shape, 32)]
    for layout in (0, 1):
        gs = [GpuConv(shape, inp, input_layout=layout) for inp in sets]
        try:
            refs = [bits(g.run()) for g in gs]
            torch.cuda.synchronize()
            for _ in range(2):
                for inp, ref in zip(sets, refs):
                    out = _run_host(gs[0], inp, True, layout)
                    assert np.array_equal(out, ref)
        finally:
            for g in gs:
                g.close()


def test_bf16_run_host_matches_device_run():
    shape = synth.CONFIGS[1]
    inp = synth.make_config_inputs_bf16(1)
    s = shape
    plan = capi.conv3d_bf16_plan(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S, s.stride, s.pad, 0)
    try:
        info = capi.conv3d_fp8_get_info(plan)
        out_shape = (s.N, s.K, info["Do"], info["Ho"], info["Wo"])
        y = torch.full(out_shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        capi.conv3d_bf16_run(plan, inp["x"].cuda(), inp["w"].cuda(), y, s.stride, s.pad)
        ref = bits(y)
        yh = torch.full(out_shape, float("nan"), dtype=torch.bfloat16).pin_memory()
        capi.conv3d_bf16_run_host(plan, inp["x"].pin_memory(), inp["w"].pin_memory(), yh,
                                  s.stride, s.pad)
        torch.cuda.synchronize()
        assert np.array_equal(bits(yh), ref)
        # the e4m3 host entry refuses a bfloat16 plan, before any copy
        sc = torch.ones(2, dtype=torch.float32)
        assert capi.conv3d_fp8_run_host_status(plan, inp["x"], inp["w"], sc, yh, s.stride,
                                               s.pad) == capi.CONV3D_EINVAL
    finally:
        capi.conv3d_fp8_destroy(plan)


def test_run_host_rejects_mismatched_stride():
    shape, inp = synth.CONFIGS[1], synth.make_config_inputs(1)
    g = GpuConv(shape, inp)
    try:
        sc = torch.tensor([inp["sx"], inp["sw"]], dtype=torch.float32)
        yh = torch.empty(g.out_shape, dtype=torch.bfloat16)
        assert capi.conv3d_fp8_run_host_status(g.plan, inp["x"], inp["w"], sc, yh, 2,
                                               shape.pad) == capi.CONV3D_EINVAL
        assert capi.conv3d_fp8_run_host_status(g.plan, inp["x"], inp["w"], None, yh,
                                               shape.stride, shape.pad) == capi.CONV3D_EINVAL
    finally:
        g.close()
