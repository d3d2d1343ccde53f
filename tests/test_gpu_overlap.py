"""The pack beside the GEMM (conv3d_fp8_options.overlap): the first input planes are packed, the
GEMM runs the whole waves of tiles that read only those while a light pack copies the other planes
beside it, and the remaining units run as a second GEMM launch -- one chain of programmatic
dependent launches on the run's stream.

Every unit is the same tile computed by the same kernel in the same K order either way, so the
output must be bit for bit the run without the overlap, for every plane count, in both input
types, on repeated runs, inside a CUDA graph (the chain's programmatic edges captured) and within
the gates against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_implicit_gemm_gb300 import capi, synth
from _gpu_common import GpuConv, GpuConvBf16, bits, check_against

pytestmark = pytest.mark.gpu


def _bits_with_and_without(cls, shape, inp, planes, repeats=1):
    on = cls(shape, inp, overlap=planes)
    off = cls(shape, inp, overlap=-1)
    try:
        assert on.info["overlap_planes"] == (planes if planes > 0 else on.info["overlap_planes"])
        assert on.info["overlap_planes"] > 0 and off.info["overlap_planes"] == 0
        ref = bits(off.run())
        outs = [bits(on.run()) for _ in range(repeats)]
        torch.cuda.synchronize()
        assert capi.conv3d_fp8_check(on.plan) == capi.CONV3D_OK
        for out in outs:
            assert np.array_equal(out, ref), f"{int(np.sum(out != ref))} outputs differ"
        return outs[0], on.info
    finally:
        on.close()
        off.close()


def test_large_layer_default_plan_overlaps_and_matches_the_single_launch():
    out, info = _bits_with_and_without(GpuConv, synth.CONFIGS[4], synth.make_config_inputs(4),
                                       0, repeats=3)
    assert (info["overlap_planes"], info["overlap_units"]) == (5, 228)


@pytest.mark.parametrize("planes", [6, 9, 15])
def test_vae_layer_plane_counts(planes):
    shape, inp = synth.CONFIGS[2], synth.make_config_inputs(2)
    out, info = _bits_with_and_without(GpuConv, shape, inp, planes)
    if planes == 6:
        y64, yb = oracle.conv3d_fp8(inp["x"].numpy(), inp["w"].numpy(), inp["sx"], inp["sw"],
                                    shape.stride, shape.pad)
        check_against(out, y64, yb, "vae layer, pack beside the GEMM")


def test_bf16_twin():
    shape = synth.CONFIGS[2]
    _bits_with_and_without(GpuConvBf16, shape, synth.make_inputs_bf16(shape, 77), 6, repeats=2)


def test_graph_capture_of_the_chain():
    shape, inp = synth.CONFIGS[2], synth.make_config_inputs(2)
    g = GpuConv(shape, inp, overlap=6)
    try:
        ref = g.run()
        y = g.new_y()
        s = torch.cuda.Stream()
        run = lambda: capi.conv3d_fp8_run(g.plan, g.x, g.w, g.sx, g.sw, y, shape.stride,
                                          shape.pad, torch.cuda.current_stream())
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            run()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run()
        y.view(torch.int16).fill_(0x7FC0)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        assert capi.conv3d_fp8_check(g.plan) == capi.CONV3D_OK
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    finally:
        g.close()
