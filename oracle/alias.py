"""Padded-row alias predictor for an implicit-GEMM conv whose epilogue guards columns only.

TEST INFRASTRUCTURE (see the package docstring for who may import it).

Source: "[Fix] conv3d fp8: guard padded M rows in the epilogue store" (ROCm/FlyDSL pull request
969), sections "Root cause" and "Verification". The M dimension (npq = N*Do*Ho*Wo output
positions) is padded up to whole tiles of TILE_M rows. For one image (n == 1) the output offset
of (row, col) is ``col * dhw + row``. A padded row (npq <= row < grid_m * TILE_M) therefore lands
on the live element of a later column whenever dhw == npq, unless the store is masked on
``row < npq``. Offsets at or beyond the end of the tensor are dropped by the hardware bound of
the buffer descriptor, so only offsets below N*K*dhw can be clobbered.

For N > 1 the page gives no formula; the general map splits row into (n, pix) with
n = row // dhw, which sends every padded row to n >= N, past the end of the tensor, so nothing
live is reachable. That reading is the one the page's remark on the other six shapes supports:
only shapes with padded rows and dhw == npq expose the race.
"""
from __future__ import annotations


def grid_m(npq: int, tile_m: int) -> int:
    return -(-npq // tile_m)


def padded_rows(npq: int, tile_m: int) -> int:
    return grid_m(npq, tile_m) * tile_m - npq


def clobberable_offsets(N: int, K: int, dhw: int, tile_m: int) -> set[int]:
    """Live output offsets a column-only-masked store of the padded rows can overwrite."""
    npq = N * dhw
    total = N * K * dhw
    rows = range(npq, grid_m(npq, tile_m) * tile_m)
    out: set[int] = set()
    if N != 1:
        return out  # general map: padded rows fall at n >= N, beyond the tensor
    for col in range(K):
        for row in rows:
            off = col * dhw + row
            if off < total:
                out.add(off)
    return out
