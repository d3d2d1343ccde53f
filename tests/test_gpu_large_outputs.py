"""An output of more than 2^31 elements: the 64-bit offsets of the stores.

y of 2 x 256 x 66 x 256 x 256 bf16 values (2.2 G elements, 4.4 GB) from an e4m3 x of 277 MB: the
epilogue's NCDHW offsets, the last image's rows and the last channels lie past 2^31 elements. The
padded-grid route on CTA pairs (the default here), the TMA im2col route on one CTA, and its TMA-store
epilogue each run into a NaN-filled y; every element must be written (no NaN left) and sampled
outputs, the ends of every image and channel among them, must meet the oracle's gates.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_implicit_gemm_gb300 import synth
from _gpu_common import GpuConv, bits, check_against, sample_indices

pytestmark = pytest.mark.gpu

SHAPE = synth.ConvShape(2, 32, 66, 256, 256, 256)


@pytest.fixture(scope="module")
def case():
    inp = synth.make_inputs(SHAPE, 8100)
    return inp


@pytest.mark.parametrize("opts", [dict(), dict(route=2, cta_pair=1),
                                  dict(route=2, cta_pair=1, epilogue=2)],
                         ids=["grid-pair", "im2col-1cta", "im2col-tma-store"])
def test_output_beyond_2_31_elements(case, opts):
    inp = case
    g = GpuConv(SHAPE, inp, **opts)
    try:
        y = g.run()
        assert y.numel() > 2 ** 31
        assert not torch.isnan(y).any().item(), "outputs left unwritten"
        idx = sample_indices(g.out_shape, 40000, 81, block_m=g.info["block_m"])
        # the last positions of every (image, channel) run of y, past 2^31 for the last image
        N, K, Do, Ho, Wo = g.out_shape
        dhw = Do * Ho * Wo
        ends = np.array([(n * K + k) * dhw + dhw - 1 - j for n in range(N) for k in (0, 1, K - 1)
                         for j in range(64)], dtype=np.int64)
        idx = np.unique(np.concatenate([idx, ends]))
        assert idx.max() > 2 ** 31
        flat = y.view(torch.int16).reshape(-1)
        got = flat[torch.from_numpy(idx).cuda()].cpu().numpy().view(np.uint16)
        y64, yb = oracle.conv3d_fp8_points(inp["x"].numpy(), inp["w"].numpy(), inp["sx"],
                                           inp["sw"], idx, SHAPE.stride, SHAPE.pad)
        check_against(got, y64, yb, f"{SHAPE} {opts}")
    finally:
        g.close()
        torch.cuda.empty_cache()
