"""Plans on separate streams at once, and a run on a non-default stream.

A plan owns its workspace, so runs of different plans may overlap on the GPU: here three plans of
three routes (padded grid on CTA pairs, TMA im2col with split-K and its reduction, the direct
route with its pre-pass) each launch many runs back to back on their own stream, with nothing
ordering the streams against each other, and every result must equal the same plan's run on the
default stream. A run is asynchronous on the stream it is given: the last test checks that its
kernels are ordered after work queued before it on that stream and before work queued after it.
"""
import numpy as np
import pytest
import torch

from fp8_implicit_gemm_gb300 import capi, synth
from _gpu_common import GpuConv, bits, NAN_BF16

pytestmark = pytest.mark.gpu

PLANS = [(synth.CONFIGS[1], {}), (synth.CONFIGS[0], dict(route=2)), (synth.CONFIGS[3], {})]


def _run_on(g: GpuConv, y: torch.Tensor, stream: torch.cuda.Stream) -> None:
    s = g.shape
    capi.conv3d_fp8_run(g.plan, g.x, g.w, g.sx, g.sw, y, s.stride, s.pad, stream)


def test_plans_overlapping_on_three_streams():
    gs = [GpuConv(shape, synth.make_inputs(shape, 7100 + i), **o)
          for i, (shape, o) in enumerate(PLANS)]
    try:
        refs = [bits(g.run()) for g in gs]
        torch.cuda.synchronize()
        streams = [torch.cuda.Stream() for _ in gs]
        reps = 20
        outs = [[g.new_y() for _ in range(reps)] for g in gs]
        torch.cuda.synchronize()
        for r in range(reps):  # interleaved launches: the streams' work can overlap
            for g, st, ys in zip(gs, streams, outs):
                _run_on(g, ys[r], st)
        torch.cuda.synchronize()
        for g, ref, ys in zip(gs, refs, outs):
            for r, y in enumerate(ys):
                assert np.array_equal(bits(y), ref), f"{g.shape}: run {r} on its own stream"
            assert capi.conv3d_fp8_check(g.plan) == capi.CONV3D_OK
    finally:
        for g in gs:
            g.close()


def test_run_is_ordered_on_its_stream():
    shape = synth.CONFIGS[1]
    g = GpuConv(shape, synth.make_inputs(shape, 7200))
    try:
        ref = bits(g.run())
        st = torch.cuda.Stream()
        y = g.new_y(0)
        torch.cuda.synchronize()  # y's allocation and zero fill are done before st touches it
        with torch.cuda.stream(st):
            y.view(torch.int16).fill_(np.int16(np.uint16(NAN_BF16).view(np.int16)))  # before
            _run_on(g, y, st)                                # must overwrite every element
            snap = y.clone()                                 # after: sees the finished run
        st.synchronize()
        assert np.array_equal(bits(snap), ref)
        assert np.array_equal(bits(y), ref)
    finally:
        g.close()
