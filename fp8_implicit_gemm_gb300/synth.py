"""Seeded synthetic inputs for the FP8 conv3d path.

This module serves both the CUDA path (tests, ``bench.py``) and the CPU oracle. It holds no
convolution arithmetic: it draws random tensors and quantises them to e4m3 bytes with a
per-tensor scale, which is how the inputs of the conv are produced, not part of the conv.

Recipe (one generator per input set, seeded; x is drawn first, then w):
  * x ~ N(0, 1), fp32, shape [N, C, D, H, W]
  * w ~ N(0, 1 / (C*T*R*S)), fp32, shape [K, C, T, R, S]
  * per-tensor scale s = amax / 448 (fp32; 1 when the tensor is all zeros);
    q = e4m3_rne(clamp(v / s, -448, 448)) through torch's float8_e4m3fn cast.
  * optional saturation: after quantising, a seeded uniform choice (without replacement) of
    floor(frac * numel) positions in each tensor is overwritten with 0x7E or 0xFE (+-448).
  No NaN byte (0x7F / 0xFF) is ever produced.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

E4M3_MAX = 448.0


@dataclass(frozen=True)
class ConvShape:
    """Problem shape: NCDHW input, KCTRS filter, isotropic or per-axis stride and padding."""
    N: int
    C: int
    D: int
    H: int
    W: int
    K: int
    T: int = 3
    R: int = 3
    S: int = 3
    stride: tuple = (1, 1, 1)
    pad: tuple = (1, 1, 1)
    sat_frac: float = 0.0
    name: str = field(default="", compare=False)

    def __post_init__(self):
        for attr in ("stride", "pad"):
            v = getattr(self, attr)
            if isinstance(v, int):
                object.__setattr__(self, attr, (v, v, v))
            else:
                object.__setattr__(self, attr, tuple(int(i) for i in v))


# The five workloads of the FP8 conv3d hot path. The first is the shape of the failing test case
# on the subject page; the other four cover n > 1, an aligned video-VAE-like block, a deep and
# narrow stride-2 layer, and a large unaligned layer with saturated values.
CONFIGS = [
    ConvShape(1, 96, 4, 8, 9, 96, name="p1_1x96x4x8x9_k96_s1 (npq=288, dhw==npq)"),
    ConvShape(2, 64, 8, 16, 15, 128, name="n2_2x64x8x16x15_k128_s1 (npq=3840)"),
    ConvShape(1, 128, 16, 64, 64, 128, name="vae_1x128x16x64x64_k128_s1 (npq=65536)"),
    ConvShape(1, 512, 4, 16, 16, 512, stride=2, name="deep_1x512x4x16x16_k512_s2 (npq=128)"),
    ConvShape(1, 256, 17, 90, 160, 256, sat_frac=0.01,
              name="large_1x256x17x90x160_k256_s1 (npq=244800, 1% saturated)"),
]


def config_seed(index: int) -> int:
    return 1000 + index


def quantize_e4m3(v: torch.Tensor) -> tuple[torch.Tensor, float]:
    """Per-tensor e4m3 quantisation: returns (uint8 bytes, fp32 scale = amax/448)."""
    v = v.float()
    amax = float(v.abs().max()) if v.numel() else 0.0
    scale = torch.tensor(amax / E4M3_MAX if amax > 0 else 1.0, dtype=torch.float32)
    q = (v / scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.contiguous(), float(scale)


def _saturate(q: torch.Tensor, frac: float, g: torch.Generator) -> None:
    m = int(frac * q.numel())
    if m <= 0:
        return
    flat = q.view(-1)
    pos = torch.randperm(flat.numel(), generator=g)[:m]
    sign = torch.randint(0, 2, (m,), generator=g, dtype=torch.uint8)
    flat[pos] = torch.where(sign.bool(), torch.tensor(0xFE, dtype=torch.uint8),
                            torch.tensor(0x7E, dtype=torch.uint8))


def make_inputs(shape: ConvShape, seed: int) -> dict:
    """Seeded e4m3 inputs on the CPU: dict(x=uint8 NCDHW, w=uint8 KCTRS, sx=float, sw=float)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn((shape.N, shape.C, shape.D, shape.H, shape.W), generator=g,
                    dtype=torch.float32)
    taps = shape.C * shape.T * shape.R * shape.S
    w = torch.randn((shape.K, shape.C, shape.T, shape.R, shape.S), generator=g,
                    dtype=torch.float32) * (1.0 / taps) ** 0.5
    xq, sx = quantize_e4m3(x)
    del x
    wq, sw = quantize_e4m3(w)
    if shape.sat_frac > 0:
        _saturate(xq, shape.sat_frac, g)
        _saturate(wq, shape.sat_frac, g)
    return {"x": xq, "w": wq, "sx": sx, "sw": sw}


def make_config_inputs(index: int) -> dict:
    return make_inputs(CONFIGS[index], config_seed(index))


def make_inputs_bf16(shape: ConvShape, seed: int) -> dict:
    """Seeded inputs of the BF16-input twin on the CPU: dict(x=bfloat16 NCDHW, w=bfloat16 KCTRS),
    x ~ N(0, 1) and w ~ N(0, 1/(C*T*R*S)) drawn in fp32 (x first) and rounded to bfloat16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn((shape.N, shape.C, shape.D, shape.H, shape.W), generator=g,
                    dtype=torch.float32).to(torch.bfloat16)
    taps = shape.C * shape.T * shape.R * shape.S
    w = (torch.randn((shape.K, shape.C, shape.T, shape.R, shape.S), generator=g,
                     dtype=torch.float32) * (1.0 / taps) ** 0.5).to(torch.bfloat16)
    return {"x": x.contiguous(), "w": w.contiguous()}


def make_config_inputs_bf16(index: int) -> dict:
    return make_inputs_bf16(CONFIGS[index], config_seed(index))


def bf16_bits(t: torch.Tensor):
    """The bit patterns of a bfloat16 CPU tensor as a numpy uint16 array."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
