"""Shared helpers of the GPU tests: run the CUDA path through the C ABI, compare with the oracle.

Tolerances (written here once, used by every parity test):
  * Frobenius: ||y_gpu - y_ref_bf16|| / ||y_ref_bf16|| <= 1e-4, against the oracle's BF16 rounding;
  * per element: |y_gpu - y64| <= 2^-7 * |y64| + 1e-3, against the oracle's unrounded fp64 value
    (one BF16 ulp is at most 2^-7 of the magnitude, so an fp32 accumulation that lands one ulp
    away still passes, a clobbered or unscaled element does not).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from fp8_implicit_gemm_gb300 import capi, synth

FROB_TOL = 1e-4
REL_TOL = 2.0 ** -7
ABS_TOL = 1e-3
# BF16-input twin. Its fp32 tensor-core accumulation of 16-bit products rounds more than the e4m3
# path's (8-bit products), so more elements land one BF16 ulp (<= 2^-7 of the magnitude) away
# from the exactly rounded value. Gate: ||g - r_bf16|| / ||r|| <= 1e-3, i.e. one-ulp flips on at
# most about (1e-3 / 2^-7)^2 = 1.6% of the elements, and ||g - y64|| / ||y64|| <= 2^-8, one BF16
# half-ulp, the most any correctly rounded result can be off in RMS. A dropped tap or a wrong
# element moves either figure by orders of magnitude; the per-element bound is unchanged.
FROB_TOL_BF16 = 1e-3
FROB64_TOL_BF16 = 2.0 ** -8
NAN_BF16 = 0x7FC0


class GpuConv:
    """A plan plus device copies of one input set."""

    def __init__(self, shape: synth.ConvShape, inp: dict, **options):
        self.shape = shape
        s = shape
        self.plan = capi.conv3d_fp8_plan(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S, s.stride,
                                         s.pad, torch.cuda.current_device(), **options)
        self.info = capi.conv3d_fp8_get_info(self.plan)
        x = inp["x"]
        if options.get("input_layout") == 1:  # the same bytes, channels-last
            x = x.permute(0, 2, 3, 4, 1).contiguous()
        self.x = x.cuda()
        self.w = inp["w"].cuda()
        self.sx = torch.tensor([inp["sx"]], dtype=torch.float32, device="cuda")
        self.sw = torch.tensor([inp["sw"]], dtype=torch.float32, device="cuda")
        self.out_shape = (s.N, s.K, self.info["Do"], self.info["Ho"], self.info["Wo"])

    def new_y(self, fill_bits: int = NAN_BF16) -> torch.Tensor:
        y = torch.empty(self.out_shape, dtype=torch.bfloat16, device="cuda")
        y.view(torch.int16).fill_(np.int16(np.uint16(fill_bits).view(np.int16)))
        return y

    def run(self, y: torch.Tensor | None = None) -> torch.Tensor:
        if y is None:
            y = self.new_y()
        capi.conv3d_fp8_run(self.plan, self.x, self.w, self.sx, self.sw, y, self.shape.stride,
                            self.shape.pad)
        return y

    def close(self):
        capi.conv3d_fp8_destroy(self.plan)
        self.plan = None


class GpuConvBf16(GpuConv):
    """A plan of the BF16-input twin plus device copies of one bfloat16 input set."""

    def __init__(self, shape: synth.ConvShape, inp: dict, **options):
        self.shape = s = shape
        self.plan = capi.conv3d_bf16_plan(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S, s.stride,
                                          s.pad, torch.cuda.current_device(), **options)
        self.info = capi.conv3d_fp8_get_info(self.plan)
        x = inp["x"]
        if options.get("input_layout") == 1:
            x = x.permute(0, 2, 3, 4, 1).contiguous()
        self.x = x.cuda()
        self.w = inp["w"].cuda()
        self.out_shape = (s.N, s.K, self.info["Do"], self.info["Ho"], self.info["Wo"])

    def run(self, y: torch.Tensor | None = None) -> torch.Tensor:
        if y is None:
            y = self.new_y()
        capi.conv3d_bf16_run(self.plan, self.x, self.w, y, self.shape.stride, self.shape.pad)
        return y


def bits(y: torch.Tensor) -> np.ndarray:
    return y.view(torch.int16).cpu().numpy().view(np.uint16)


def check_against(gpu_bits: np.ndarray, y64: np.ndarray, ref_bits: np.ndarray, what: str = "",
                  frob_tol: float = FROB_TOL, frob64_tol: float | None = None):
    """Assert the gates (Frobenius against the oracle's BF16 rounding, per element against its
    fp64 value, optionally Frobenius against fp64); returns the measured errors."""
    g = oracle.bf16_bits_to_f64(gpu_bits).ravel()
    r = oracle.bf16_bits_to_f64(ref_bits).ravel()
    y64 = np.asarray(y64, dtype=np.float64).ravel()
    n_nan = int(np.isnan(g).sum())
    assert n_nan == 0, f"{what}: {n_nan} outputs never written (NaN pre-fill left)"
    denom = np.linalg.norm(r)
    frob = float(np.linalg.norm(g - r) / denom) if denom > 0 else float(np.linalg.norm(g - r))
    bound = REL_TOL * np.abs(y64) + ABS_TOL
    viol = np.abs(g - y64) > bound
    zeroed = int(np.sum((g == 0) & (y64 != 0) & (np.abs(y64) > bound)))
    assert zeroed == 0, f"{what}: {zeroed} live outputs zeroed"
    assert not viol.any(), (f"{what}: {int(viol.sum())} elements beyond |d| <= 2^-7|ref| + 1e-3; "
                            f"worst at {int(np.argmax(np.abs(g - y64) - bound))}")
    assert frob <= frob_tol, f"{what}: Frobenius relative error {frob:.3e} > {frob_tol}"
    if frob64_tol is not None:
        d64 = np.linalg.norm(y64)
        frob64 = float(np.linalg.norm(g - y64) / d64) if d64 > 0 else float(np.linalg.norm(g))
        assert frob64 <= frob64_tol, f"{what}: Frobenius vs fp64 {frob64:.3e} > {frob64_tol}"
    flips = int(np.sum(gpu_bits.ravel() != ref_bits.ravel()))
    return {"frob": frob, "bf16_flips": flips, "n": g.size}


def sample_indices(out_shape, count: int, seed: int, block_m: int = 128) -> np.ndarray:
    """Random flat NCDHW indices plus the structured ones most likely to expose an index bug:
    the first and last output positions of every image, the padded-tile edge (the last
    block_m rows of the GEMM view), faces of the volume, and first/last channels."""
    N, K, Do, Ho, Wo = out_shape
    dhw = Do * Ho * Wo
    total = N * K * dhw
    rng = np.random.default_rng(seed)
    idx = [rng.integers(0, total, count)]
    npq = N * dhw
    last_rows = np.arange(max(0, npq - 2 * block_m), npq)
    for col in (0, 1, K // 2, K - 1):
        n = last_rows // dhw
        idx.append((n * K + col) * dhw + last_rows % dhw)
        first = np.arange(0, min(npq, 2 * block_m))
        idx.append((first // dhw * K + col) * dhw + first % dhw)
    # every 6-face of the first image for a few channels
    d, h, w = np.meshgrid(np.arange(Do), np.arange(Ho), np.arange(Wo), indexing="ij")
    face = (d == 0) | (d == Do - 1) | (h == 0) | (h == Ho - 1) | (w == 0) | (w == Wo - 1)
    fpix = (d * Ho * Wo + h * Wo + w)[face]
    for col in (0, K - 1):
        for n in {0, N - 1}:
            idx.append((n * K + col) * dhw + fpix[:4096])
    out = np.unique(np.concatenate(idx).astype(np.int64))
    return out[(out >= 0) & (out < total)]
