"""Helper of tests/test_gpu_write_count.py, run in a process of its own: it loads the
write-counting build of the library (C3D_COUNT_WRITES) in place of the product build and, for each
case, counts the stores to every output element over one run. Prints one line per case and exits
non-zero when any element was written other than exactly once."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import torch  # noqa: E402

from fp8_implicit_gemm_gb300 import build, capi, synth  # noqa: E402

build.LIB_PATH = build.build_counting()

# (name, shape, plan options, x source): every route and kernel, whole and split tiles, the
# split-K reduction, the TMA-store epilogue (whole tiles, rows spilling into the next image), a
# channels-last x, and a run that quantises its x
CASES = [
    ("grid-pair, tail split", synth.ConvShape(1, 256, 8, 10, 12, 256),
     dict(route=3, cta_pair=2, max_ctas=8), "e4m3"),
    ("grid-pair, two images", synth.CONFIGS[1], dict(), "e4m3"),
    ("im2col-1cta, every tile split", synth.CONFIGS[0], dict(route=2), "e4m3"),
    ("im2col-pair", synth.CONFIGS[0], dict(route=2, cta_pair=2, splits=1), "e4m3"),
    ("gather-1cta, odd shape", synth.ConvShape(2, 48, 4, 6, 5, 80), dict(route=1), "e4m3"),
    ("direct-1cta, split-K", synth.CONFIGS[3], dict(), "e4m3"),
    ("TMA-store epilogue, images in a tile", synth.ConvShape(9, 48, 2, 3, 4, 40),
     dict(route=1, epilogue=2, splits=1), "e4m3"),
    ("TMA-store epilogue on pairs", synth.ConvShape(2, 64, 4, 6, 5, 80),
     dict(route=2, cta_pair=2, epilogue=2, splits=1), "e4m3"),
    ("channels-last x, grid", synth.CONFIGS[1], dict(input_layout=1), "e4m3"),
    ("fp32 x quantised in the pack", synth.CONFIGS[1], dict(), "fp32"),
    ("vae layer", synth.CONFIGS[2], dict(), "e4m3"),
    ("large layer (tail split over 18 units, pack beside the GEMM)", synth.CONFIGS[4], dict(),
     "e4m3"),
    ("vae layer, pack beside the GEMM from plane 6", synth.CONFIGS[2], dict(overlap=6), "e4m3"),
]


def main() -> int:
    bad = 0
    for name, shape, opts, src in CASES:
        s = shape
        inp = synth.make_inputs(s, 4242)
        plan = capi.conv3d_fp8_plan(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S, s.stride, s.pad,
                                    0, **opts)
        try:
            info = capi.conv3d_fp8_get_info(plan)
            out_shape = (s.N, s.K, info["Do"], info["Ho"], info["Wo"])
            counts = torch.zeros(out_shape, dtype=torch.int32, device="cuda")
            st = capi.conv3d_fp8_set_write_counter_status(plan, counts)
            assert st == capi.CONV3D_OK, st
            y = torch.full(out_shape, float("nan"), dtype=torch.bfloat16, device="cuda")
            w = inp["w"].cuda()
            sw = torch.tensor([inp["sw"]], dtype=torch.float32, device="cuda")
            if src == "fp32":
                g = torch.Generator().manual_seed(77)
                xf = torch.randn((s.N, s.C, s.D, s.H, s.W), generator=g).cuda()
                capi.conv3d_fp8_run_quantize_x(plan, xf, w, sw, y, s.stride, s.pad)
            else:
                x = inp["x"]
                if opts.get("input_layout") == 1:
                    x = x.permute(0, 2, 3, 4, 1).contiguous()
                sx = torch.tensor([inp["sx"]], dtype=torch.float32, device="cuda")
                capi.conv3d_fp8_run(plan, x.cuda(), w, sx, sw, y, s.stride, s.pad)
            torch.cuda.synchronize()
            ok_status = capi.conv3d_fp8_check(plan) == capi.CONV3D_OK
            n = counts.numel()
            ones = int((counts == 1).sum().item())
            lo, hi = int(counts.min().item()), int(counts.max().item())
            nan_left = int(torch.isnan(y).sum().item())
            good = ones == n and ok_status and nan_left == 0
            bad += 0 if good else 1
            print(f"{'ok ' if good else 'BAD'} {name}: {n} elements, counts in [{lo}, {hi}], "
                  f"{n - ones} not written exactly once, NaN left {nan_left}, plan route "
                  f"{info['route']} pair {info['cta_pair']} epilogue {info['epilogue']} "
                  f"splits {info['splits']} whole tiles {info['full_tiles']} overlap "
                  f"{info['overlap_planes']}/{info['overlap_units']}", flush=True)
        finally:
            capi.conv3d_fp8_destroy(plan)
    return 1 if bad else 0


if __name__ == "__main__":
    sys.exit(main())
