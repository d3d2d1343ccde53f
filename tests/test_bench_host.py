"""Host-side arithmetic of bench.py, on the CPU: problem figures (GEMM view, FLOP, bytes), the
roofline bound and fraction, and the algorithmic bytes of the operand re-layout per route."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from fp8_implicit_gemm_gb300 import build, capi, synth  # noqa: E402


def test_problem_figures_match_the_workloads():
    figs = [bench.problem_figures(s) for s in synth.CONFIGS]
    assert [f["npq"] for f in figs] == [288, 3840, 65536, 128, 244800]
    assert [f["k_gemm"] for f in figs] == [2592, 1728, 3456, 13824, 6912]
    # FLOP = 2 npq K K_gemm, padding taps counted
    assert figs[2]["flop"] == 2.0 * 65536 * 128 * 3456
    assert round(figs[4]["flop"] / 1e9, 1) == 866.3
    # bytes: x and w in e4m3 (one byte), y in bf16
    s = synth.CONFIGS[4]
    assert figs[4]["x_bytes"] == s.N * s.C * s.D * s.H * s.W
    assert figs[4]["w_bytes"] == s.K * s.C * 27
    assert figs[4]["y_bytes"] == 2 * 244800 * 256
    assert figs[4]["alg_bytes"] == figs[4]["x_bytes"] + figs[4]["w_bytes"] + figs[4]["y_bytes"]
    # the BF16 twin's inputs take two bytes an element
    b = bench.problem_figures(s, 2)
    assert b["x_bytes"] == 2 * figs[4]["x_bytes"] and b["w_bytes"] == 2 * figs[4]["w_bytes"]


def test_roofline_picks_the_slower_bound():
    fp8, hbm = 3859.2, 6685.1
    big = bench.problem_figures(synth.CONFIGS[4])
    deep = bench.problem_figures(synth.CONFIGS[3])
    r = bench.roofline_of(big, 0.2298, fp8, hbm)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(big["flop"] / 0.2298e-3 / 1e12, rel=1e-3)
    assert r["frac"] == pytest.approx(r["achieved"] / fp8, abs=1e-4)
    r = bench.roofline_of(deep, 0.0164, fp8, hbm)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(deep["alg_bytes"] / 0.0164e-3 / 1e9, rel=1e-3)
    # a time at the roofline reads a fraction of one
    t_roof_ms = max(big["flop"] / (fp8 * 1e12), big["alg_bytes"] / (hbm * 1e9)) * 1e3
    assert bench.roofline_of(big, t_roof_ms, fp8, hbm)["frac"] == pytest.approx(1.0, abs=1e-3)


def test_pack_bytes_per_route():
    big = bench.problem_figures(synth.CONFIGS[4])
    deep = bench.problem_figures(synth.CONFIGS[3])
    # transpose of x plus the weight re-layout: each read once and written once
    assert bench.pack_alg_bytes(big, True) == 2 * big["x_bytes"] + 2 * big["w_bytes"]
    # a channels-last x read by TMA directly: only the weights move
    assert bench.pack_alg_bytes(big, False) == 2 * big["w_bytes"]
    # direct route: x read, the explicit im2col (npq x K_gemm elements) written, weights untouched
    assert bench.pack_alg_bytes(deep, True, 4) == deep["x_bytes"] + 128 * 13824
    assert bench.pack_alg_bytes(deep, True, 4, 2) == deep["x_bytes"] + 2 * 128 * 13824


def test_overlap_splits_the_pack_bytes():
    # the large layer packs 5 of 17 planes (rounded up to whole 256-position tiles) before the
    # GEMM and the rest beside it: the two parts add up to the whole pack
    build.build()  # host-only planning through the library (no GPU needed)
    s = synth.CONFIGS[4]
    fig = bench.problem_figures(s)
    info = capi.conv3d_fp8_describe(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S, s.stride,
                                    s.pad, 152)
    first, beside = bench.overlap_pack_bytes(fig, s, info)
    assert first + beside == bench.pack_alg_bytes(fig, True, 3)
    q_a = 72192  # 5 * 90 * 160 = 72000 positions, rounded up to a multiple of 256
    assert first == 2 * fig["w_bytes"] + 2 * 256 * q_a
    assert bench.overlap_pack_bytes(fig, s, dict(info, overlap_planes=0)) is None
    assert "two launches" in bench.gemm_label(info)


def test_pack_kernel_names_follow_the_library_rule():
    # the tiled transpose takes an NCDHW x with W % 4 == 0, D*H*W*bytes % 16 == 0, C % 64 == 0
    names = [bench.pack_kernel_name(s, 3, False, False, False) for s in synth.CONFIGS]
    assert names == ["pack_kernel", "pack_kernel", "pack_x_transpose_kernel",
                     "pack_x_transpose_kernel", "pack_x_transpose_kernel"]
    large = synth.CONFIGS[4]
    assert bench.pack_kernel_name(large, 3, False, True, False) == "pack_x_transpose_kernel"
    assert bench.pack_kernel_name(large, 3, False, False, True) == "pack_kernel"  # weights only
    assert bench.pack_kernel_name(large, 4, False, False, False) == "im2col_kernel"
    assert bench.pack_kernel_name(large, 3, True, False, False).startswith("pack_x_tiled_kernel")


def test_both_arms_print_the_same_config():
    # the reference arm (the CPU oracle) runs on the GPU arm's workload: one config builder serves
    # both, and nothing in it depends on the run (plan, buffer sizes and timings live elsewhere)
    import argparse
    import json
    import subprocess

    args = argparse.Namespace(dtype="e4m3", quantize_x=None, input_layout="ncdhw")
    shape = synth.CONFIGS[0]
    cfg = bench.bench_config(shape, bench.problem_figures(shape), args, 1)
    assert cfg["workload"] == shape.name and cfg["npq"] == 288 and "plan" not in cfg
    assert cfg["parallelism"] == "replicas x1" and cfg["l2"].startswith("flushed between steps")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--config", "0", "--steps", "2", "--warmup", "1", "--ref-seconds", "1"],
                         capture_output=True, text=True, timeout=600, cwd=root,
                         env={**os.environ, "WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["config"] == cfg
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s"
