"""A run captured into a CUDA graph and replayed: the same bits as a direct run, and the scales
are read on the device at replay time (changing them between replays changes the output).

The run's launches carry programmatic-dependent-launch attributes; stream capture records them as
graph edges, so a replay keeps the overlap of each kernel's prologue with its predecessor.
"""
import pytest
import torch

from fp8_implicit_gemm_gb300 import capi, synth
from _gpu_common import GpuConv, GpuConvBf16

pytestmark = pytest.mark.gpu

CASES = [0, 1, 3]  # every-tile split (reduction launched), whole tiles on pairs, one-CTA kernel


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm the plan's host-side state (tensor maps) outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("cfg", CASES)
def test_graph_replay_matches_direct_run(cfg):
    shape = synth.CONFIGS[cfg]
    inp = synth.make_config_inputs(cfg)
    g = GpuConv(shape, inp)
    try:
        ref = g.run()
        y = g.new_y()
        graph = _capture(lambda: capi.conv3d_fp8_run(g.plan, g.x, g.w, g.sx, g.sw, y,
                                                      shape.stride, shape.pad,
                                                      torch.cuda.current_stream()))
        y.view(torch.int16).fill_(0x7FC0)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        assert capi.conv3d_fp8_check(g.plan) == capi.CONV3D_OK
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
        # the scales are device data: doubling sw between replays doubles every output exactly
        g.sw.mul_(2.0)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y.float(), 2.0 * ref.float())
    finally:
        g.close()


def test_graph_replay_bf16_twin():
    shape = synth.CONFIGS[1]
    inp = synth.make_inputs_bf16(shape, 41)
    g = GpuConvBf16(shape, inp)
    try:
        ref = g.run()
        y = g.new_y()
        graph = _capture(lambda: capi.conv3d_bf16_run(g.plan, g.x, g.w, y, shape.stride,
                                                       shape.pad, torch.cuda.current_stream()))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    finally:
        g.close()
