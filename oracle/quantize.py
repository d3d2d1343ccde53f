"""CPU oracle of the per-tensor e4m3 quantiser (the "fp8cast" producer of the e4m3 bytes).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this module; the CUDA package imports nothing from it.

What it computes. The subject page ("[Fix] conv3d fp8: guard padded M rows in the epilogue store",
section "Problem") checks the kernel against an "fp8cast reference": e4m3 inputs made from real
values with a per-tensor scale. The page prints no formula; the reading used here (the plainest
one, also the harness's): with v the fp32 values of one tensor,

    amax  = max |v|
    s     = fp32(amax / 448)            (448 = the largest finite e4m3 value; s = 1 when amax == 0)
    q[i]  = e4m3_rne(clamp(fp32(v[i] / s), -448, 448))

fp32(a / b) is IEEE fp32 division (round to nearest even). It is computed here in float64 and
rounded once to fp32: for two 24-bit operands a 53-bit quotient holds at least 2 * 24 + 2 bits, so
rounding it to 24 bits gives the correctly rounded quotient (double rounding is innocuous at that
width; the pins check it against exact rational arithmetic). e4m3_rne rounds to the nearest value
of the e4m3 grid (3 mantissa bits, exponent bias 7, subnormal spacing 2^-9), ties to the even code.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def scale_of(amax) -> np.float32:
    """fp32(amax / 448), or 1 for an all-zero tensor."""
    a = np.float32(amax)
    if a == 0:
        return np.float32(1.0)
    return np.float32(np.float64(a) / E4M3_MAX)


def fp32_div(v, s) -> np.ndarray:
    """IEEE fp32 quotient v / s of fp32 operands (correctly rounded, via one float64 division)."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    return (v / np.float64(np.float32(s))).astype(np.float32)


def e4m3_rne(r) -> np.ndarray:
    """Round fp32 values in [-448, 448] to the e4m3 grid, ties to even; returns the byte codes."""
    r = np.asarray(r, dtype=np.float64)
    if np.any(np.abs(r) > E4M3_MAX) or np.any(np.isnan(r)):
        raise ValueError("e4m3_rne: value outside [-448, 448]")
    sign = np.signbit(r)
    a = np.abs(r)
    # exponent of the binade holding a (normal range: a >= 2^-6); below it the subnormal spacing
    _, e = np.frexp(a)              # a = f * 2^e with f in [0.5, 1)
    e = e - 1                       # a in [2^e, 2^(e+1))
    e = np.maximum(e, -6)           # 2^-6 is the smallest normal; below it the spacing stays 2^-9
    quantum = np.ldexp(1.0, e - 3)  # 3 mantissa bits
    k = np.rint(a / quantum)        # round half to even (exact: a / quantum is a power-of-two rescale)
    mag = k * quantum
    # encode: normal  = (8 + m) * 2^(E - 10), E in 1..15; subnormal = m * 2^-9 (E = 0)
    code = np.zeros(a.shape, dtype=np.uint8)
    sub = mag < 2.0 ** -6
    code[sub] = (mag[sub] / 2.0 ** -9).astype(np.uint8)
    nm = ~sub
    _, ee = np.frexp(mag[nm])
    E = ee - 1 + 7                  # biased exponent of the rounded value
    M = mag[nm] / np.ldexp(1.0, ee - 1) * 8 - 8
    code[nm] = (E.astype(np.int64) << 3 | M.astype(np.int64)).astype(np.uint8)
    code[sign] |= 0x80
    return code


def quantize(v):
    """Quantise one tensor of fp32 values: returns (uint8 e4m3 codes, fp32 scale)."""
    v = np.asarray(v, dtype=np.float32)
    amax = np.float32(np.max(np.abs(v))) if v.size else np.float32(0)
    s = scale_of(amax)
    r = np.clip(fp32_div(v, s), -E4M3_MAX, E4M3_MAX)
    return e4m3_rne(r), s


def quantize_points(v, idx, s):
    """The codes of the elements at flat indices ``idx`` for a given scale (sampled checks)."""
    v = np.asarray(v, dtype=np.float32).ravel()[np.asarray(idx, dtype=np.int64)]
    return e4m3_rne(np.clip(fp32_div(v, s), -E4M3_MAX, E4M3_MAX))
