#!/usr/bin/env python
"""Benchmark of the FP8 (e4m3) implicit-GEMM conv3d on one GB300, through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config I] [--impl ours|reference]

A step is one conv3d_fp8_run (operand packing, the tcgen05 implicit-GEMM kernel and, for
split-K plans, the ordered reduction) over one batch of seeded synthetic e4m3 inputs already
resident in HBM. The default workload is the largest single-GPU layer of the five (1x256x17x90x160
-> 256 channels, 3x3x3, stride 1, pad 1: 866 GFLOP); ``--config`` picks another.

Metric: TFLOP/s, FLOP = 2 * N*Do*Ho*Wo * K * C*T*R*S (padding taps counted). L2 is flushed
between steps by a 2x-L2-sized write that lies outside the per-step CUDA events.

Multi-GPU: the path needs no exchange, so N GPUs run N independent replicas of the same workload
(weak scaling); ranks meet only at the barriers that bracket the timed region, and the slowest
rank's time is the job's time.

``--impl reference`` times the CPU oracle (fp64, OpenMP) on rank 0 on bounded samples of the
same workload; the other ranks exit without work.

Prints exactly one JSON line on stdout (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_CONFIG = 4
# --route: the planner's choice, or one route forced (conv3d_fp8_options.route)
ROUTES = {"auto": 0, "gather": 1, "im2col": 2, "grid": 3, "direct": 4}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0  # nominal dense fp8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)
METRIC = "conv3d fp8 TFLOP/s and % of FP8/HBM roofline at 1 GB300"
METRIC_BF16 = "conv3d BF16-input twin TFLOP/s and % of BF16/HBM roofline at 1 GB300"
DATA = "synthetic (seeded N(0,1) inputs quantised to e4m3 per tensor)"
DATA_BF16 = "synthetic (seeded N(0,1) inputs rounded to bfloat16)"
MAIN_KERNEL_SOURCES = ["conv_tc.cu", "conv_tc_pair.cu", "conv_common.cuh", "ptx.cuh",
                       "conv3d_fp8_internal.h"]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------------- problem math
def problem_figures(shape, elem_bytes: int = 1):
    Do = (shape.D + 2 * shape.pad[0] - shape.T) // shape.stride[0] + 1
    Ho = (shape.H + 2 * shape.pad[1] - shape.R) // shape.stride[1] + 1
    Wo = (shape.W + 2 * shape.pad[2] - shape.S) // shape.stride[2] + 1
    npq = shape.N * Do * Ho * Wo
    kg = shape.C * shape.T * shape.R * shape.S
    flop = 2.0 * npq * shape.K * kg
    x_bytes = elem_bytes * shape.N * shape.C * shape.D * shape.H * shape.W
    w_bytes = elem_bytes * shape.K * kg
    y_bytes = 2 * npq * shape.K
    return {"Do": Do, "Ho": Ho, "Wo": Wo, "npq": npq, "k_gemm": kg, "flop": flop,
            "x_bytes": x_bytes, "w_bytes": w_bytes, "y_bytes": y_bytes,
            "alg_bytes": x_bytes + w_bytes + y_bytes}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def main_kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in MAIN_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "fp8_implicit_gemm_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str, input_layout: str = "NCDHW", overlap_planes: int = 0):
    """DRAM bytes of the main kernel in one step from a committed ncu summary, if that summary was
    taken on the current kernel source for this workload, input layout and plane count of the
    pack beside the GEMM (line: ``bench-traffic: {json}``; a line without "input_layout" is an
    NCDHW capture, one without "overlap_planes" a single GEMM launch). With the overlap the two
    GEMM launches of a step are summed ("dram_bytes_per_step")."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    want = main_kernel_source_hash()
    for name in sorted(os.listdir(pdir)):
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, name)) as f:
            for line in f:
                if line.startswith("bench-traffic:"):
                    try:
                        d = json.loads(line.split(":", 1)[1])
                    except ValueError:
                        continue
                    if (d.get("workload") == workload and d.get("source_sha256") == want and
                            d.get("input_layout", "NCDHW") == input_layout and
                            d.get("overlap_planes", 0) == overlap_planes):
                        return d.get("dram_bytes_per_step", d.get("dram_bytes_per_launch"))
    return None


# --------------------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id is not None:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self, min_samples: int = 2, wait_s: float = 1.0):
        if self.proc is None:
            return
        t0 = time.time()
        while len(self.lines) < min_samples and time.time() - t0 < wait_s:
            time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self):
        if self.proc is None or not self.lines:
            return None
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_query_id(torch, dev: int):
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = getattr(props, "pci_bus_id", None)
        dom = getattr(props, "pci_domain_id", 0)
        pdev = getattr(props, "pci_device_id", 0)
        if bus is not None:
            return f"{dom:08x}:{bus:02x}:{pdev:02x}.0"
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if dev < len(ids):
            return ids[dev]
    return str(dev)


# --------------------------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Dist:
    def __init__(self, backend: str):
        import torch.distributed as dist
        self.dist = dist
        self.world, self.rank, self.local = dist_env()
        self.on = self.world > 1
        if self.on and not dist.is_initialized():
            dist.init_process_group(backend=backend)

    def barrier(self):
        if self.on:
            self.dist.barrier()

    def max(self, v: float, device=None) -> float:
        if not self.on:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.on and self.dist.is_initialized():
            self.dist.destroy_process_group()


# ------------------------------------------------------------------------------- CPU baseline
def oracle_points_fn(inp, shape, bf16: bool):
    """The oracle's sampled-points call on this input set (e4m3 with scales, or the BF16 twin)."""
    import oracle
    from fp8_implicit_gemm_gb300 import synth
    if bf16:
        x, w = synth.bf16_bits(inp["x"]), synth.bf16_bits(inp["w"])
        return lambda idx: oracle.conv3d_bf16_points(x, w, idx, shape.stride, shape.pad)
    x, w = inp["x"].numpy(), inp["w"].numpy()
    return lambda idx: oracle.conv3d_fp8_points(x, w, inp["sx"], inp["sw"], idx, shape.stride,
                                                shape.pad)


def cpu_oracle_sample(inp, shape, target_s: float, seed: int, min_points: int = 256,
                      bf16: bool = False):
    """Time the oracle on a random sample of outputs sized to about target_s seconds."""
    import numpy as np
    import oracle
    fig = problem_figures(shape)
    total = shape.K * fig["npq"]
    points = oracle_points_fn(inp, shape, bf16)
    rng = np.random.default_rng(seed)
    n = min_points
    t = 0.0
    while True:
        idx = rng.integers(0, total, n)
        t0 = time.perf_counter()
        points(idx)
        t = time.perf_counter() - t0
        if t >= target_s * 0.5 or n >= total:
            break
        n = int(min(total, max(n * 2, n * target_s / max(t, 1e-3))))
    flop = 2.0 * fig["k_gemm"] * n
    return {"value": flop / t / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle", "seconds": round(t, 3),
            "sample": f"{n} random outputs of {total} (fp64 direct sum, one by one)"}


# ------------------------------------------------------------------------------ per workload
def pack_alg_bytes(fig, packs_x: bool, route: int = 0, elem_bytes: int = 1) -> int:
    """Compulsory bytes of the operand re-layout: the weights read and written once, and x read
    and its channels-last interior written once when the run transposes x. On the direct route
    (4) the weights stay as they are and the pre-pass reads x and writes the explicit im2col of
    x once (npq rows of C*T*R*S elements)."""
    if route == 4:
        return fig["x_bytes"] + elem_bytes * fig["npq"] * fig["k_gemm"]
    return 2 * fig["w_bytes"] + (2 * fig["x_bytes"] if packs_x else 0)


PACK_TILE_POSITIONS = 256  # the library rounds the first pack's positions up to this


def overlap_pack_bytes(fig, shape, info, elem_bytes: int = 1):
    """With the pack beside the GEMM (plan info overlap_planes > 0): the compulsory bytes of the
    pack before the GEMM (the weights, and x's first planes read and written) and of the light
    pack beside it (the rest of x read and written). None without the overlap."""
    planes = info.get("overlap_planes", 0)
    if not planes:
        return None
    hw, dhw_in = shape.H * shape.W, shape.D * shape.H * shape.W
    q_a = min(dhw_in, -(-planes * hw // PACK_TILE_POSITIONS) * PACK_TILE_POSITIONS)
    x_first = fig["x_bytes"] * q_a // dhw_in
    return 2 * fig["w_bytes"] + 2 * x_first, 2 * (fig["x_bytes"] - x_first)


def gemm_label(info) -> str:
    k = "conv3d_fp8_tc_pair_kernel" if info["cta_pair"] == 2 else "conv3d_fp8_tc_kernel"
    if info.get("overlap_planes", 0):
        k += " (two launches) + pack_x_transpose_kernel beside the first"
    if info["full_tiles"] < info["m_tiles"] * info["n_tiles"]:
        # the timed window then also holds the reduction of the tiles split along K
        k += " + splitk_reduce_kernel"
    return k


def roofline_of(fig, kernel_ms: float, fp8_peak: float, hbm_peak: float) -> dict:
    """Roofline of one launch: the slower of the dense tensor rate and HBM bandwidth for the
    algorithmic FLOP and bytes (x + w + y once), against the measured kernel time."""
    t_flop = fig["flop"] / (fp8_peak * 1e12)
    t_hbm = fig["alg_bytes"] / (hbm_peak * 1e9)
    s = kernel_ms * 1e-3
    if t_flop >= t_hbm:
        ach = fig["flop"] / s / 1e12
        return {"bound": "tensor", "achieved": round(ach, 1), "peak": round(fp8_peak, 1),
                "unit": "TFLOP/s", "frac": round(ach / fp8_peak, 4)}
    ach = fig["alg_bytes"] / s / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": round(hbm_peak, 1),
            "unit": "GB/s", "frac": round(ach / hbm_peak, 4)}


def measure_config(index: int, inp, dev, stream, flush, fp8_peak: float, hbm_peak: float,
                   steps: int = 100, warmup: int = 5) -> dict:
    """One workload's default e4m3 plan: step time (events around each run), main-kernel time and
    pack time (the library's events), TFLOP/s and the roofline fraction. L2 is flushed before
    every step; medians over `steps` steps."""
    import torch
    from fp8_implicit_gemm_gb300 import capi, synth

    shape = synth.CONFIGS[index]
    fig = problem_figures(shape)
    if inp is None:
        inp = synth.make_config_inputs(index)
    plan = capi.conv3d_fp8_plan(shape.N, shape.C, shape.D, shape.H, shape.W, shape.K, shape.T,
                                shape.R, shape.S, shape.stride, shape.pad, dev)
    try:
        info = capi.conv3d_fp8_get_info(plan)
        x, w = inp["x"].to(dev), inp["w"].to(dev)
        sx = torch.tensor([inp["sx"]], dtype=torch.float32, device=dev)
        sw = torch.tensor([inp["sw"]], dtype=torch.float32, device=dev)
        y = torch.full((shape.N, shape.K, fig["Do"], fig["Ho"], fig["Wo"]), float("nan"),
                       dtype=torch.bfloat16, device=dev)

        def run():
            capi.conv3d_fp8_run(plan, x, w, sx, sw, y, shape.stride, shape.pad, stream)

        for _ in range(warmup):
            flush.fill_(3)
            run()
        torch.cuda.synchronize()
        if torch.isnan(y).any().item():
            raise RuntimeError(f"{shape.name}: outputs left unwritten")
        mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        ev = [(mk(), mk()) for _ in range(steps)]
        for i in range(steps):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            run()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        step = [a.elapsed_time(b) for a, b in ev]
        evk = [(mk(), mk(), mk()) for _ in range(steps)]
        for e in evk:
            for e_ in e:
                e_.record(stream)
        torch.cuda.synchronize()
        for i in range(steps):
            flush.fill_(i & 0xFF)
            capi.conv3d_fp8_set_pack_timing_event(plan, evk[i][0])
            capi.conv3d_fp8_set_timing_events(plan, evk[i][1], evk[i][2])
            run()
        torch.cuda.synchronize()
        capi.conv3d_fp8_set_pack_timing_event(plan, None)
        capi.conv3d_fp8_set_timing_events(plan, None, None)
        if capi.conv3d_fp8_check(plan) != capi.CONV3D_OK:
            raise RuntimeError(f"{shape.name}: a kernel reported a timed-out wait")
        kern = [b.elapsed_time(c) for _, b, c in evk]
        pack = [a.elapsed_time(b) for a, b, _ in evk]
    finally:
        capi.conv3d_fp8_destroy(plan)
    k_ms, s_ms, p_ms = (statistics.median(kern), statistics.median(step),
                        statistics.median(pack))
    roof = roofline_of(fig, k_ms, fp8_peak, hbm_peak)
    step_roof = roofline_of(fig, s_ms, fp8_peak, hbm_peak)
    pbytes = pack_alg_bytes(fig, True, info["route"])
    ov = overlap_pack_bytes(fig, shape, info)
    if ov:
        pbytes = ov[0]
    return {
        "workload": shape.name, "config_index": index,
        "plan": {k: info[k] for k in ("route", "cta_pair", "block_m", "block_n", "m_tiles",
                                      "n_tiles", "full_tiles", "splits", "stages", "grid",
                                      "overlap_planes", "overlap_units")},
        "gflop": round(fig["flop"] / 1e9, 4), "alg_bytes": fig["alg_bytes"],
        "kernel": gemm_label(info),
        "kernel_ms": round(k_ms, 5), "kernel_ms_min": round(min(kern), 5),
        "kernel_ms_mean": round(statistics.mean(kern), 5),
        "step_ms": round(s_ms, 5), "step_ms_min": round(min(step), 5),
        "step_ms_mean": round(statistics.mean(step), 5),
        "pack_ms": round(p_ms, 5),
        "kernel_tflops": round(fig["flop"] / (k_ms * 1e-3) / 1e12, 2),
        "step_tflops": round(fig["flop"] / (s_ms * 1e-3) / 1e12, 2),
        "kernel_gbs": round(fig["alg_bytes"] / (k_ms * 1e-3) / 1e9, 1),
        "step_gbs": round(fig["alg_bytes"] / (s_ms * 1e-3) / 1e9, 1),
        "roofline": roof, "step_roofline_frac": step_roof["frac"],
        "pack": {"kernel": pack_kernel_name(shape, info["route"], False, False, False),
                 "alg_bytes": pbytes, "ms": round(p_ms, 5),
                 "achieved_gbs": round(pbytes / (p_ms * 1e-3) / 1e9, 1),
                 "frac_of_hbm": round(pbytes / (p_ms * 1e-3) / 1e9 / hbm_peak, 4),
                 "beside_gemm_bytes": ov[1] if ov else 0},
        "steps": steps, "timing": "medians (means beside them: the event clock ticks in ~1 us "
                                  "steps); CUDA events on the launching stream; L2 flushed before "
                                  "every step",
    }


# ----------------------------------------------------------------------------------------- ours
def run_ours(args):
    import numpy as np
    import torch
    from fp8_implicit_gemm_gb300 import build, capi, synth

    dist = Dist("nccl")
    torch.cuda.set_device(dist.local)
    dev = torch.cuda.current_device()
    build.build()
    shape = synth.CONFIGS[args.config]
    bf16 = args.dtype == "bf16"  # the BF16-input twin instead of the e4m3 path
    fig = problem_figures(shape, 2 if bf16 else 1)
    inp = synth.make_config_inputs_bf16(args.config) if bf16 else synth.make_config_inputs(args.config)
    channels_last = args.input_layout == "ndhwc"
    # the library's x: the same bytes, laid out NDHWC when asked (the oracle keeps NCDHW)
    x_lib = inp["x"].permute(0, 2, 3, 4, 1).contiguous() if channels_last else inp["x"]
    quant = args.quantize_x  # x handed over as fp32 / bf16 values, quantised on the device
    if quant:
        if bf16 or channels_last:
            raise SystemExit("--quantize-x runs the e4m3 path on an NCDHW x")
        g = torch.Generator().manual_seed(synth.config_seed(args.config))
        x_lib = torch.randn((shape.N, shape.C, shape.D, shape.H, shape.W), generator=g).to(
            torch.float32 if quant == "fp32" else torch.bfloat16)

    make_plan = capi.conv3d_bf16_plan if bf16 else capi.conv3d_fp8_plan
    plan = make_plan(shape.N, shape.C, shape.D, shape.H, shape.W, shape.K, shape.T, shape.R,
                     shape.S, shape.stride, shape.pad, dev, input_layout=1 if channels_last else 0,
                     route=ROUTES[args.route], overlap=args.overlap)
    info = capi.conv3d_fp8_get_info(plan)
    stream = torch.cuda.current_stream()
    x = x_lib.to(dev)
    w = inp["w"].to(dev)
    sx = torch.tensor([inp.get("sx", 1.0)], dtype=torch.float32, device=dev)
    sw = torch.tensor([inp.get("sw", 1.0)], dtype=torch.float32, device=dev)
    y = torch.full((shape.N, shape.K, fig["Do"], fig["Ho"], fig["Wo"]), float("nan"),
                   dtype=torch.bfloat16, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    # pack, main kernel, and the reduction when some tiles are split along K (+ the amax
    # reduction and the scale finalisation when x is quantised on the device)
    launches_per_step = 2 + (1 if info["full_tiles"] < info["m_tiles"] * info["n_tiles"] else 0)
    launches_per_step += 2 if quant else 0
    # the pack beside the GEMM: a second GEMM launch and the light pack
    launches_per_step += 2 if (info.get("overlap_planes", 0) and not quant) else 0

    def run(scale_x, scale_w):
        if quant:
            capi.conv3d_fp8_run_quantize_x(plan, x, w, scale_w, y, shape.stride, shape.pad, None,
                                           stream)
        elif bf16:
            capi.conv3d_bf16_run(plan, x, w, y, shape.stride, shape.pad, stream)
        else:
            capi.conv3d_fp8_run(plan, x, w, scale_x, scale_w, y, shape.stride, shape.pad, stream)

    def step():
        run(sx, sw)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if torch.isnan(y).any().item():
        raise RuntimeError("outputs left unwritten after warm-up")
    capi.conv3d_fp8_check(plan)

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for e in ev:  # materialise the lazily created events before they are handed to the library
        for x_ in e:
            x_.record()
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_query_id(torch, dev))
    sampler.start()
    time.sleep(0.3)
    dist.barrier()
    torch.cuda.synchronize()
    # The steps are timed as a user runs them: CUDA events on the stream around each step only. The
    # library's own events around the implicit GEMM (the roofline's kernel time) sit between its
    # kernels and hold back their programmatic dependent launches, so they are recorded in a
    # second timed pass of the same steps.
    t_wall0 = time.perf_counter()
    for i in range(K):
        flush.fill_(i & 0xFF)
        s0, s1 = ev[i][0], ev[i][1]
        s0.record(stream)
        step()
        s1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    t_wall = time.perf_counter() - t_wall0
    K2 = min(K, 500)  # kernel-time pass
    for i in range(K2):
        flush.fill_(i & 0xFF)
        capi.conv3d_fp8_set_pack_timing_event(plan, ev[i][4])
        capi.conv3d_fp8_set_timing_events(plan, ev[i][2], ev[i][3])
        step()
    torch.cuda.synchronize()
    sampler.stop()
    capi.conv3d_fp8_set_pack_timing_event(plan, None)
    capi.conv3d_fp8_set_timing_events(plan, None, None)
    if capi.conv3d_fp8_check(plan) != capi.CONV3D_OK:
        raise RuntimeError("a kernel reported a timed-out wait")
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    kern_ms = [ev[i][2].elapsed_time(ev[i][3]) for i in range(K2)]
    pack_ms = [ev[i][4].elapsed_time(ev[i][2]) for i in range(K2)]
    # L2-warm figure (reported beside the headline, not instead of it): the same steps back to
    # back without the flush, so each step finds the previous step's operands in L2
    K3 = min(K, 500)
    for i in range(K3):
        s0, s1 = ev[i][0], ev[i][1]
        s0.record(stream)
        step()
        s1.record(stream)
    torch.cuda.synchronize()
    warm_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K3)]
    total_ms = dist.max(sum(step_ms), dev)
    mean_step_ms = total_ms / K
    mean_kern_ms = statistics.mean(kern_ms)
    value = fig["flop"] * K * dist.world / (total_ms * 1e-3) / 1e12

    # ---- end to end through the public C-ABI call with host buffers. Every step copies its inputs
    # from page-locked host memory and its result back. The e4m3 and bfloat16 runs go through the
    # host-buffer entry point (conv3d_fp8_run_host / conv3d_bf16_run_host: the copies in, the run
    # and the copy out, enqueued by one call); as a user would, consecutive steps are pipelined by
    # rotating three plans on three streams, so that one step's copy in, another's run and a third's
    # copy out can overlap (with two, a stream's next copy in waits for its own copy out). The
    # quantising run has no host-buffer entry: its copies go by torch on streams of their own,
    # around conv3d_fp8_run_quantize_x on device buffers (two buffer sets).
    x_h = x_lib.pin_memory()
    w_h = inp["w"].pin_memory()
    # host scales of the e4m3 path (the BF16 twin has none)
    s_h = torch.tensor([inp["sx"], inp["sw"]] if not bf16 else [1.0, 1.0],
                       dtype=torch.float32).pin_memory()
    nbuf = 2
    xs = [x] + [torch.empty_like(x) for _ in range(nbuf - 1)]
    ws = [w] + [torch.empty_like(w) for _ in range(nbuf - 1)]
    ss = [torch.empty(2, dtype=torch.float32, device=dev) for _ in range(nbuf)]
    ys = [y] + [torch.empty_like(y) for _ in range(nbuf - 1)]
    yhs = [torch.empty(y.shape, dtype=torch.bfloat16).pin_memory() for _ in range(nbuf)]
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    e2e_steps = max(3, min(K, 200))

    def ev():
        return torch.cuda.Event(enable_timing=True)

    e_start, e_stop = ev(), ev()
    if quant:
        api = "conv3d_fp8_run_quantize_x (device buffers; copies by torch)"
        pipelining = "H2D / compute / D2H of consecutive steps on three streams, two buffer sets"
        ev_h2d = [ev() for _ in range(e2e_steps)]
        ev_comp = [ev() for _ in range(e2e_steps)]
        ev_d2h = [ev() for _ in range(e2e_steps)]
        torch.cuda.synchronize()
        dist.barrier()
        e_start.record(h2d_stream)
        for i in range(e2e_steps):
            b = i % nbuf
            with torch.cuda.stream(h2d_stream):  # inputs of step i, once step i - nbuf read them
                if i >= nbuf:
                    h2d_stream.wait_event(ev_comp[i - nbuf])
                xs[b].copy_(x_h, non_blocking=True)
                ws[b].copy_(w_h, non_blocking=True)
                ss[b].copy_(s_h, non_blocking=True)
                ev_h2d[i].record(h2d_stream)
            stream.wait_event(ev_h2d[i])          # step i computes after its inputs arrived and
            if i >= nbuf:                         # after step i - nbuf's result left its buffer
                stream.wait_event(ev_d2h[i - nbuf])
            capi.conv3d_fp8_run_quantize_x(plan, xs[b], ws[b], ss[b][1:2], ys[b], shape.stride,
                                           shape.pad, None, stream)
            ev_comp[i].record(stream)
            with torch.cuda.stream(d2h_stream):  # the result of step i back to the host
                d2h_stream.wait_event(ev_comp[i])
                yhs[b].copy_(ys[b], non_blocking=True)
                ev_d2h[i].record(d2h_stream)
        e_stop.record(d2h_stream)
    else:
        api = "conv3d_bf16_run_host" if bf16 else "conv3d_fp8_run_host"
        nhost = 3
        pipelining = (f"consecutive steps rotate over {nhost} plans on {nhost} streams; a step's "
                      "H2D copies, run and D2H copy are one host-buffer call")
        plans = [plan] + [make_plan(shape.N, shape.C, shape.D, shape.H, shape.W, shape.K, shape.T,
                                    shape.R, shape.S, shape.stride, shape.pad, dev,
                                    input_layout=1 if channels_last else 0,
                                    route=ROUTES[args.route], overlap=args.overlap)
                          for _ in range(nhost - 1)]
        host_streams = [stream] + [torch.cuda.Stream() for _ in range(nhost - 1)]
        yhs = [torch.empty(y.shape, dtype=torch.bfloat16).pin_memory() for _ in range(nhost)]

        def run_host(b):
            if bf16:
                capi.conv3d_bf16_run_host(plans[b], x_h, w_h, yhs[b], shape.stride, shape.pad,
                                          host_streams[b])
            else:
                capi.conv3d_fp8_run_host(plans[b], x_h, w_h, s_h, yhs[b], shape.stride,
                                         shape.pad, host_streams[b])

        for b in range(nhost):  # each plan's first call allocates its device buffers: untimed
            run_host(b)
        torch.cuda.synchronize()
        for yh in yhs:
            yh.fill_(float("nan"))
        dist.barrier()
        e_start.record(host_streams[0])
        for hs in host_streams[1:]:
            hs.wait_event(e_start)
        for i in range(e2e_steps):
            run_host(i % nhost)
        for hs in host_streams[1:]:
            host_streams[0].wait_stream(hs)
        e_stop.record(host_streams[0])
    torch.cuda.synchronize()
    e2e_ms = dist.max(e_start.elapsed_time(e_stop) / e2e_steps, dev)
    dist.barrier()
    if not quant:
        for pl in plans:
            if capi.conv3d_fp8_check(pl) != capi.CONV3D_OK:
                raise RuntimeError("a host-buffer run reported a timed-out wait")
        for pl in plans[1:]:
            capi.conv3d_fp8_destroy(pl)
    if any(torch.isnan(t.float()).any().item() for t in yhs):
        raise RuntimeError("e2e result has unwritten outputs")
    e2e = {"value": fig["flop"] * dist.world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "ms_per_step": round(e2e_ms, 4),
           "h2d_bytes_per_step": int(x_h.numel() * x_h.element_size() +
                                     w_h.numel() * w_h.element_size() +
                                     (0 if bf16 else 4 * s_h.numel())),
           "d2h_bytes_per_step": int(2 * y.numel()),
           "api": api, "pipelining": pipelining}
    # The host link's floor under the pipelined step: the same bytes moved in both directions at
    # once (the step's H2D copies on one stream, its D2H copy on the other) with nothing else
    # running, timed after the e2e loop. The pipelined e2e step cannot beat it.
    link_reps = 5
    for i in range(link_reps + 2):
        if i == 2:
            torch.cuda.synchronize()
            l_start, l_stop = ev(), ev()
            l_start.record(stream)
        h2d_stream.wait_stream(stream)
        d2h_stream.wait_stream(stream)
        with torch.cuda.stream(h2d_stream):
            xs[0].copy_(x_h, non_blocking=True)
            ws[0].copy_(w_h, non_blocking=True)
            ss[0].copy_(s_h, non_blocking=True)
        with torch.cuda.stream(d2h_stream):
            yhs[0].copy_(ys[0], non_blocking=True)
        stream.wait_stream(h2d_stream)
        stream.wait_stream(d2h_stream)
    l_stop.record(stream)
    torch.cuda.synchronize()
    link_ms = dist.max(l_start.elapsed_time(l_stop) / link_reps, dev)
    e2e["link_floor"] = {
        "ms_per_step": round(link_ms, 4),
        "gbs": round((e2e["h2d_bytes_per_step"] + e2e["d2h_bytes_per_step"]) /
                     (link_ms * 1e-3) / 1e9, 1),
        "frac": round(link_ms / e2e_ms, 4),
        "note": "the step's H2D and D2H bytes copied at once, alone, on the same streams; frac = "
                "this floor / the e2e step"}

    # ---- roofline of the dominant kernel (the implicit-GEMM kernel)
    peaks, peaks_kind = load_peaks()
    # the contraction's own dtype: e4m3 = the measured bf16 peak x the nominal fp8/bf16 ratio
    fp8_peak = (1.0 if bf16 else FP8_PER_BF16) * float(peaks["bf16_tflops"])
    hbm_peak = float(peaks["hbm_gbs"])
    t_flop = fig["flop"] / (fp8_peak * 1e12)
    t_hbm = fig["alg_bytes"] / (hbm_peak * 1e9)
    workload = shape.name + (" [bf16 inputs]" if bf16 else "")
    traffic = committed_traffic(workload, "NDHWC" if channels_last else "NCDHW",
                                0 if quant else info.get("overlap_planes", 0))
    if t_flop >= t_hbm:
        achieved = fig["flop"] / (mean_kern_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(fp8_peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 4),
                "peak_source": (f"{peaks_kind} bf16 burst" if bf16 else
                                f"{peaks_kind} bf16 burst x {FP8_PER_BF16:g} (nominal fp8/bf16)")}
    else:
        achieved = fig["alg_bytes"] / (mean_kern_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": round(hbm_peak, 1),
                "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                "peak_source": f"{peaks_kind} copy bandwidth"}
    roof["traffic"] = traffic
    ov_active = bool(info.get("overlap_planes", 0)) and not quant
    roof["kernel"] = gemm_label(info if ov_active else dict(info, overlap_planes=0))
    roof["kernel_ms"] = round(mean_kern_ms, 5)
    roof["kernel_timing"] = (f"library events around the GEMM (+ reduce) on the launching stream, "
                             f"{K2} steps after the {K} timed ones")
    roof["alg_flop"] = fig["flop"]
    roof["alg_bytes"] = fig["alg_bytes"]
    roof["step_roofline_frac"] = round(max(t_flop, t_hbm) / (mean_step_ms * 1e-3), 4)
    # the operand re-layout of the same steps (HBM-bound): the pack alone, by the library's events
    packs_x = not channels_last or info["route"] == 1
    if not quant:
        p_bytes = pack_alg_bytes(fig, packs_x, info["route"], 2 if bf16 else 1)
    elif info["route"] == 4:  # the pre-pass quantises x into the explicit im2col
        p_bytes = x.numel() * x.element_size() + fig["npq"] * fig["k_gemm"]
    else:
        p_bytes = 2 * fig["w_bytes"] + x.numel() * x.element_size() + fig["x_bytes"]
    ov = overlap_pack_bytes(fig, shape, info, 2 if bf16 else 1) if ov_active else None
    if ov:
        p_bytes = ov[0]
    p_ms = statistics.mean(pack_ms)
    pack = {"kernel": pack_kernel_name(shape, info["route"], quant, bf16, channels_last),
            "alg_bytes": int(p_bytes), "ms": round(p_ms, 5),
            "achieved": round(p_bytes / (p_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "peak": round(hbm_peak, 1), "frac": round(p_bytes / (p_ms * 1e-3) / 1e9 / hbm_peak, 4),
            "timing": "library events before the pack and before the main kernel, same steps as "
                      "kernel_ms"}
    if ov:
        pack["beside_gemm"] = {
            "alg_bytes": int(ov[1]),
            "note": "the other input planes, packed by the light pack_x_transpose_kernel beside "
                    "the first GEMM launch: inside kernel_ms, not in this record's ms or bytes"}

    # ---- every workload's default e4m3 plan (NCDHW x), one record each
    per_config = None
    if not bf16 and not quant and not channels_last and not args.no_per_config:
        per_config = []
        for ci in range(len(synth.CONFIGS)):
            per_config.append(measure_config(ci, inp if ci == args.config else None, dev, stream,
                                             flush, fp8_peak, hbm_peak))

    # ---- the device quantiser alone (two passes over x: amax, then the cast), HBM-bound
    quantiser = None
    if quant:
        n = x.numel()
        qdst = torch.empty(n, dtype=torch.uint8, device=dev)
        qscale = torch.empty(1, dtype=torch.float32, device=dev)
        qms = []
        for i in range(13):
            flush.fill_(i & 255)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            capi.conv3d_fp8_quantize(x, qdst, qscale, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                qms.append(e0.elapsed_time(e1))
        qbytes = 2 * n * x.element_size() + n  # read x twice (amax, cast), write the codes
        q_ms = statistics.median(qms)
        quantiser = {"kernels": "amax_kernel + quant_cast_kernel + quant_finalize_kernel",
                     "bound": "hbm", "ms": round(q_ms, 5), "alg_bytes": qbytes,
                     "achieved": round(qbytes / (q_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                     "peak": round(hbm_peak, 1),
                     "frac": round(qbytes / (q_ms * 1e-3) / 1e9 / hbm_peak, 4)}

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(inp, shape, args.cpu_seconds, seed=7, bf16=bf16)

    clocks = sampler.summary()
    capi.conv3d_fp8_destroy(plan)
    out = {
        "metric": METRIC_BF16 if bf16 else METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": dist.world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(mean_step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if bf16 else "e4m3",
        "data": DATA_BF16 if bf16 else DATA,
        "config": bench_config(shape, fig, args, dist.world),
        "plan": {k: info[k] for k in ("route", "cta_pair", "block_m", "block_n", "m_tiles",
                                      "n_tiles", "full_tiles", "splits", "stages", "grid",
                                      "row_chk", "overlap_planes", "overlap_units")},
        "roofline": roof,
        "pack": pack,
        "per_config": per_config,
        "quantiser": quantiser,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "wall_s_timed_region": round(t_wall, 3),
        "step_ms_stats": {"min": round(min(step_ms), 5),
                          "median": round(statistics.median(step_ms), 5),
                          "max": round(max(step_ms), 5)},
        "l2_warm": {"steps": K3, "ms_per_step_median": round(statistics.median(warm_ms), 5),
                    "value": round(fig["flop"] / (statistics.median(warm_ms) * 1e-3) / 1e12, 2),
                    "note": "no flush between steps; outside the timed region"},
    }
    if dist.rank == 0:
        print(json.dumps(out), flush=True)
    dist.close()


# ------------------------------------------------------------------------------------ reference
def pack_kernel_name(shape, route: int, quant: bool, bf16: bool, channels_last: bool) -> str:
    """The kernel the library launches in front of the GEMM for this run (its choice, restated)."""
    if route == 4:
        return "im2col_kernel"
    if quant:
        return "pack_x_tiled_kernel + pack items"
    dhw = shape.D * shape.H * shape.W
    eb = 2 if bf16 else 1
    if not channels_last and shape.W % 4 == 0 and (dhw * eb) % 16 == 0 and shape.C % 64 == 0:
        return "pack_x_transpose_kernel"
    return "pack_kernel"


def bench_config(shape, fig, args, world: int) -> dict:
    """The workload of a bench line, the same for both arms: the layer, its input form, the L2
    treatment between the GPU arm's steps and the replica count."""
    bf16 = args.dtype == "bf16"
    quant = args.quantize_x
    return {"workload": shape.name + (" [bf16 inputs]" if bf16 else ""), "N": shape.N,
            "C": shape.C, "D": shape.D, "H": shape.H, "W": shape.W, "K": shape.K,
            "filter": [shape.T, shape.R, shape.S], "stride": list(shape.stride),
            "pad": list(shape.pad), "npq": fig["npq"],
            "gflop_per_step": round(fig["flop"] / 1e9, 3),
            "input_layout": "NDHWC" if args.input_layout == "ndhwc" else "NCDHW",
            "output_layout": "NCDHW",
            "x_source": (f"{quant} values, quantised to e4m3 on the device every step"
                         if quant else ("bfloat16 values" if bf16 else "e4m3 bytes")),
            "l2": "flushed between steps (a write of at least twice the L2 size, outside the "
                  "per-step events)",
            "parallelism": f"replicas x{world}"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from fp8_implicit_gemm_gb300 import synth

    oracle.build()
    shape = synth.CONFIGS[args.config]
    bf16 = args.dtype == "bf16"
    fig = problem_figures(shape, 2 if bf16 else 1)
    inp = synth.make_config_inputs_bf16(args.config) if bf16 else synth.make_config_inputs(args.config)
    points = oracle_points_fn(inp, shape, bf16)
    total = shape.K * fig["npq"]
    rng = np.random.default_rng(11)
    # size each step so that warm-up + timed steps take about args.ref_seconds in total
    probe = rng.integers(0, total, 512)
    t0 = time.perf_counter()
    points(probe)
    rate = 512 / max(time.perf_counter() - t0, 1e-6)
    per_step = max(32, int(rate * args.ref_seconds / max(1, args.steps + args.warmup)))
    per_step = min(per_step, total)
    for _ in range(args.warmup):
        points(rng.integers(0, total, per_step))
    times = []
    for _ in range(args.steps):
        idx = rng.integers(0, total, per_step)
        t0 = time.perf_counter()
        points(idx)
        times.append(time.perf_counter() - t0)
    flop = 2.0 * fig["k_gemm"] * per_step
    ms = 1e3 * statistics.mean(times)
    value = flop * len(times) / sum(times) / 1e12
    sample = f"{per_step} random outputs of {total} per step (fp64 direct sum, one by one)"
    out = {
        "impl": "reference",
        "metric": METRIC_BF16 if bf16 else METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": DATA_BF16 if bf16 else DATA,
        "config": bench_config(shape, fig, args, world),
        "oracle_run": "rank 0 only, the CPU oracle on the host cores",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload records (every config's default e4m3 plan)")
    ap.add_argument("--dtype", choices=["e4m3", "bf16"], default="e4m3",
                    help="input type: the e4m3 path, or its BF16-input twin")
    ap.add_argument("--quantize-x", choices=["fp32", "bf16"], default=None,
                    help="hand x over as fp32 / bf16 values: each step quantises it on the device")
    ap.add_argument("--route", choices=list(ROUTES), default="auto",
                    help="how A reaches the tensor cores: the library's choice, or one route forced")
    ap.add_argument("--overlap", type=int, default=0,
                    help="conv3d_fp8_options.overlap: 0 the library's choice, -1 never, P > 0 "
                         "pack P input planes before the GEMM starts")
    ap.add_argument("--input-layout", choices=["ncdhw", "ndhwc"], default="ncdhw",
                    help="layout of x handed to the library (y is NCDHW either way)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, _, _ = dist_env()
    if world != args.gpus:
        log(f"note: --gpus {args.gpus} but WORLD_SIZE={world}; using WORLD_SIZE")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
