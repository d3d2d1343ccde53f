"""Every output element written exactly once, counted directly.

The NaN pre-fill of the other tests shows that every element is written at least once and that
no launch clobbers another's values; a second store of the same value would pass it. Here the
write-counting build of the library (C3D_COUNT_WRITES: every store to y also adds one to a
per-element counter) runs every route and kernel, split tiles and their reduction, the TMA-store
epilogue and a quantising run, and every counter must end at exactly 1. It runs in a process of
its own (tests/_write_count_run.py), so that the counting library is the only one loaded there.
The product build refuses the counter (EUNSUPPORTED), so the product never counts.
"""
import os
import subprocess
import sys

import pytest
import torch

from fp8_implicit_gemm_gb300 import capi, synth

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_every_element_written_exactly_once():
    r = subprocess.run([sys.executable, os.path.join(HERE, "_write_count_run.py")],
                       capture_output=True, text=True, timeout=1200)
    print(r.stdout)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    assert r.stdout.count("ok ") >= 13


def test_product_build_does_not_count():
    s = synth.CONFIGS[0]
    plan = capi.conv3d_fp8_plan(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S, s.stride, s.pad, 0)
    try:
        counts = torch.zeros(16, dtype=torch.int32, device="cuda")
        assert capi.conv3d_fp8_set_write_counter_status(plan, counts) == capi.CONV3D_EUNSUPPORTED
    finally:
        capi.conv3d_fp8_destroy(plan)
