"""C-ABI checks that need no GPU: the library loads, exports every declared entry point, and its
host-only planning and validation behave as documented in include/conv3d_fp8.h."""
import ctypes
import os
import re

import pytest

from fp8_implicit_gemm_gb300 import build, capi, synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "conv3d_fp8.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return capi.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(conv3d_(?:fp8|bf16)_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("conv3d_fp8_plan", "conv3d_fp8_run", "conv3d_fp8_destroy",
              "conv3d_fp8_workspace_size", "conv3d_fp8_strerror", "conv3d_fp8_run_host",
              "conv3d_bf16_plan", "conv3d_bf16_run", "conv3d_bf16_run_host"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_strerror(lib):
    for code in range(6):
        assert capi.conv3d_fp8_strerror(code)
    assert "unknown" in capi.conv3d_fp8_strerror(99)


def _describe(shape, sm=152, **kw):
    return capi.conv3d_fp8_describe(shape.N, shape.C, shape.D, shape.H, shape.W, shape.K, shape.T,
                                    shape.R, shape.S, shape.stride, shape.pad, sm, **kw)


def test_describe_configs(lib):
    infos = [_describe(s) for s in synth.CONFIGS]
    npq = [i["npq"] for i in infos]
    # stride 2 on 4x16x16 with pad 1 gives a 2x8x8 output: npq = 128
    assert npq == [288, 3840, 65536, 128, 244800]
    assert [i["k_gemm"] for i in infos] == [2592, 1728, 3456, 13824, 6912]
    # stride-1 layers whose padded output grid adds at most 30% rows take the padded-grid route,
    # on CTA pairs (256-row tiles); the deep layer (one 128-row tile, 512 output channels) the
    # direct route on one CTA (the weights are read as they are); the first layer the TMA im2col
    # route on one CTA
    assert [i["cta_pair"] for i in infos] == [1, 2, 2, 1, 2]
    assert [i["block_m"] for i in infos] == [128, 256, 256, 128, 256]
    assert [i["route"] for i in infos] == [2, 3, 3, 4, 3]
    # grid route: N * ceil(Do*Hp*Wp / 256) tiles, (t, r, channel block) groups as K blocks
    assert [i["m_tiles"] for i in infos] == [3, 2 * 10, 273, 1, 990]
    assert [i["k_blocks"] for i in infos] == [21, 9, 9, 108, 18]
    assert [i["row_chk"] for i in infos] == [1, 1, 1, 0, 1]
    assert [i["block_n"] for i in infos] == [96, 128, 128, 256, 256]
    single = [_describe(s, cta_pair=1) for s in synth.CONFIGS]
    assert [i["m_tiles"] for i in single] == [3, 30, 512, 1, 1913]
    assert [i["row_chk"] for i in single] == [1, 0, 0, 0, 1]
    for i in infos:
        assert i["grid"] % (2 if i["cta_pair"] == 2 else 1) == 0
    # deep and narrow -> every tile split along K; the 65536-position layer fills its waves well
    # enough to compute every tile whole
    assert infos[3]["splits"] > 1 and infos[3]["full_tiles"] == 0
    assert infos[2]["splits"] == 1 and infos[2]["full_tiles"] == infos[2]["m_tiles"]
    for i in infos:
        kb = i["k_blocks"]
        assert i["splits"] * i["k_blocks_per_split"] >= kb
        assert (i["splits"] - 1) * i["k_blocks_per_split"] < kb  # no empty split
        assert i["grid"] <= 152 and i["stages"] >= 3
        assert i["workspace_bytes"] > 0


def test_describe_routes(lib):
    # every workload has C % 32 == 0 and unit paddings: TMA im2col unless the padded grid applies
    assert all(_describe(s, route=2)["route"] == 2 for s in synth.CONFIGS)
    assert capi.conv3d_fp8_describe_status(1, 512, 4, 16, 16, 512, 3, 3, 3, 2, 1, 152,
                                           route=3) == capi.CONV3D_EUNSUPPORTED  # stride 2
    assert capi.conv3d_fp8_describe_status(1, 128, 4, 8, 8, 64, 3, 3, 3, 1, 1, 152, route=3,
                                           cta_pair=1) == capi.CONV3D_EUNSUPPORTED  # one CTA
    assert _describe(synth.CONFIGS[0], route=3)["route"] == 3
    odd = synth.ConvShape(1, 48, 8, 8, 8, 16)                   # npq > K: not direct
    assert _describe(odd)["route"] == 1                         # C % 32 != 0 -> gather
    assert capi.conv3d_fp8_describe_status(1, 48, 4, 4, 4, 16, 3, 3, 3, 1, 1, 152,
                                           route=2) == capi.CONV3D_EUNSUPPORTED
    assert _describe(synth.CONFIGS[0], route=1)["route"] == 1   # forced gather
    big_pad = synth.ConvShape(1, 32, 4, 4, 4, 16, pad=17)       # corner beyond [-16, 15]
    assert _describe(big_pad, cta_pair=1)["route"] == 1          # im2col impossible -> gather
    assert _describe(big_pad)["route"] == 3                      # the padded grid takes any pad
    # the gather and padded-grid routes' packed copy carries the zero halo, the im2col one not
    s = synth.CONFIGS[2]
    ws = {r: _describe(s, route=r, splits=1)["workspace_bytes"] for r in (1, 2, 3)}
    assert ws[1] > ws[2] and ws[3] == ws[1]


def test_describe_direct_route(lib):
    # any NCDHW shape can be forced onto it; it runs on one CTA, re-lays no weights (its
    # workspace holds the explicit im2col of x, npq rows of C*T*R*S bytes, instead) and keeps
    # K_gemm in the KCTRS order of the caller's weights
    for s in synth.CONFIGS:
        i = _describe(s, route=4)
        kg = s.C * s.T * s.R * s.S
        assert i["route"] == 4 and i["cta_pair"] == 1 and i["block_m"] == 128
        assert i["k_blocks"] == -(-kg // 128)
        assert i["workspace_bytes"] >= i["npq"] * kg
    deep = synth.CONFIGS[3]
    w_bytes = deep.K * deep.C * 27
    a_bytes = 128 * deep.C * 27
    assert (_describe(deep, route=2)["workspace_bytes"] - _describe(deep, route=4)["workspace_bytes"]
            >= w_bytes - a_bytes)
    # not with a channels-last x, not on CTA pairs
    assert capi.conv3d_fp8_describe_status(1, 512, 4, 16, 16, 512, 3, 3, 3, 2, 1, 152, route=4,
                                           input_layout=1) == capi.CONV3D_EUNSUPPORTED
    assert capi.conv3d_fp8_describe_status(1, 512, 4, 16, 16, 512, 3, 3, 3, 2, 1, 152, route=4,
                                           cta_pair=2) == capi.CONV3D_EUNSUPPORTED
    # by default only for small GEMMs (at most four 128-row tiles) with no more output positions
    # than output channels (the explicit A is then no bigger than the weights)
    assert _describe(synth.ConvShape(1, 512, 4, 16, 16, 512, stride=2))["route"] == 4
    assert _describe(synth.ConvShape(1, 512, 4, 16, 16, 64, stride=2))["route"] == 2  # npq > K
    assert _describe(synth.ConvShape(1, 512, 8, 32, 32, 512, stride=2))["route"] == 2  # npq 2048


def test_describe_pair_rules(lib):
    odd = synth.ConvShape(1, 48, 4, 4, 4, 16)                      # gather route: no pairs
    assert _describe(odd)["cta_pair"] == 1
    assert capi.conv3d_fp8_describe_status(1, 48, 4, 4, 4, 16, 3, 3, 3, 1, 1, 152,
                                           cta_pair=2) == capi.CONV3D_EUNSUPPORTED
    i = _describe(synth.CONFIGS[3], cta_pair=2)                    # forced on a single tile
    assert i["cta_pair"] == 2 and i["m_tiles"] == 1 and i["row_chk"] == 1
    assert _describe(synth.CONFIGS[4], cta_pair=1)["route"] == 2   # no grid route on one CTA
    i = _describe(synth.CONFIGS[4], max_ctas=9)                    # pairs round the cap down
    assert i["grid"] == 8


def test_describe_tail_split(lib):
    # large layer on 76 CTA pairs: 990 tiles = 13 full waves + 2 tiles; those 2 are split along K
    # over the idle pairs of the last wave (18 groups of taps: one per split, 36 units)
    i = _describe(synth.CONFIGS[4])
    assert i["full_tiles"] == 13 * 76 and i["splits"] == 18 and i["k_blocks_per_split"] == 1
    units = i["full_tiles"] + (i["m_tiles"] * i["n_tiles"] - i["full_tiles"]) * i["splits"]
    assert units == 13 * 76 + 36 and i["grid"] == 152
    assert i["workspace_bytes"] >= 36 * 256 * 256 * 4               # fp32 partials of the tail
    # a CTA cap changes the waves: 75 pairs -> 13 waves + 15 tiles, split 5 ways (4 groups each)
    i = _describe(synth.CONFIGS[4], max_ctas=150)
    assert i["full_tiles"] == 13 * 75 and i["splits"] == 5 and i["k_blocks_per_split"] == 4
    # a last wave more than half full is left alone (one CTA per tile: 1913 = 12 * 152 + 89)
    i = _describe(synth.CONFIGS[4], cta_pair=1)
    assert i["full_tiles"] == i["m_tiles"] == 1913 and i["splits"] == 1
    # few tiles: every tile split, down to three K blocks a split when the K loop is short (the
    # p1 layer: 21 blocks in 7 splits), four otherwise (the deep layer: 108 blocks in 27; its
    # bfloat16 twin: 216 in 54)
    p1 = _describe(synth.CONFIGS[0])
    assert (p1["splits"], p1["k_blocks_per_split"], p1["full_tiles"]) == (7, 3, 0)
    deep = _describe(synth.CONFIGS[3])
    assert (deep["splits"], deep["k_blocks_per_split"]) == (27, 4)
    s3 = synth.CONFIGS[3]
    deep2 = capi.conv3d_bf16_describe(s3.N, s3.C, s3.D, s3.H, s3.W, s3.K, s3.T, s3.R, s3.S,
                                      s3.stride, s3.pad, 152)
    assert (deep2["splits"], deep2["k_blocks_per_split"]) == (54, 4)
    # a split count in the options applies to every tile
    assert _describe(synth.CONFIGS[4], splits=1)["full_tiles"] == 990
    i = _describe(synth.CONFIGS[4], splits=3)
    assert i["full_tiles"] == 0 and i["splits"] == 3
    # a short K loop is not worth a reduction: 546 tiles of 9 groups of 6 N = 128 MMAs (~3500
    # tensor cycles a tile) keep their 14-tile tail whole
    short = synth.ConvShape(2, 64, 16, 64, 64, 128)
    i = _describe(short)
    assert i["m_tiles"] * i["n_tiles"] == 546 and i["splits"] == 1
    assert _describe(short, max_ctas=150)["splits"] == 1


def test_describe_pack_beside_gemm(lib):
    # the large layer (13 whole waves): the first 5 planes packed first, 3 waves of tiles read only
    # those; the rest of x is packed beside them, the other units run as a second launch
    i = _describe(synth.CONFIGS[4])
    assert (i["overlap_planes"], i["overlap_units"]) == (5, 3 * 76)
    s4 = synth.CONFIGS[4]
    b = capi.conv3d_bf16_describe(s4.N, s4.C, s4.D, s4.H, s4.W, s4.K, s4.T, s4.R, s4.S,
                                  s4.stride, s4.pad, 152)
    assert (b["overlap_planes"], b["overlap_units"]) == (5, 3 * 76)
    # off on request; a chosen plane count runs the whole waves of tiles those planes feed
    assert _describe(s4, overlap=-1)["overlap_planes"] == 0
    assert (_describe(s4, overlap=3)["overlap_units"], _describe(s4, overlap=16)["overlap_units"]) \
        == (76, 11 * 76)
    # none by default under four whole waves (the vae layer: 273 tiles on 76 pairs), where a plane
    # count can still ask for it; never on the other routes, with a channels-last x or 2 images
    assert _describe(synth.CONFIGS[2])["overlap_planes"] == 0
    assert (_describe(synth.CONFIGS[2], overlap=6)["overlap_units"]) == 76
    for cfg in (0, 1, 3):
        assert _describe(synth.CONFIGS[cfg])["overlap_planes"] == 0
    assert _describe(s4, input_layout=1)["overlap_planes"] == 0
    two = synth.ConvShape(2, 256, 17, 90, 160, 256)
    assert _describe(two)["overlap_planes"] == 0
    # a plane count that feeds no whole wave, or leaves nothing to pack beside the GEMM, or a
    # shape the overlap cannot take, is refused
    for bad, opts in ((s4, dict(overlap=2)), (s4, dict(overlap=17)), (two, dict(overlap=5)),
                      (s4, dict(overlap=5, input_layout=1)), (s4, dict(overlap=-2))):
        st = capi.conv3d_fp8_describe_status(bad.N, bad.C, bad.D, bad.H, bad.W, bad.K, bad.T,
                                             bad.R, bad.S, bad.stride, bad.pad, 152, **opts)
        assert st == (capi.CONV3D_EINVAL if opts.get("overlap") == -2
                      else capi.CONV3D_EUNSUPPORTED), (bad, opts, st)


def _overlap_reads_and_writes(shape, info):
    """Padded planes the first GEMM launch reads (the last tile's last row plus the farthest tap)
    and the first padded plane the light pack writes, from the plan's figures alone."""
    pd, ph, pw = shape.pad
    Hg, Wg = shape.H + 2 * ph, shape.W + 2 * pw
    reach = (shape.T - 1) * Hg * Wg + (shape.R - 1) * Wg + (shape.S - 1)
    last_m = (info["overlap_units"] - 1) // info["n_tiles"]
    last_row = info["block_m"] * (last_m + 1) - 1 + reach
    hw = shape.H * shape.W
    q_a = min(shape.D * hw, -(-info["overlap_planes"] * hw // 256) * 256)
    return last_row // (Hg * Wg), pd + q_a // hw, q_a


@pytest.mark.parametrize("shape", [synth.CONFIGS[4], synth.CONFIGS[2],
                                   synth.ConvShape(1, 128, 33, 128, 128, 128),
                                   synth.ConvShape(1, 64, 20, 40, 256, 192)])
def test_overlap_first_launch_reads_only_packed_planes(lib, shape):
    # for every plane count the planner accepts: the first launch's tiles read only padded planes
    # that the first pack completed, the light pack writes only planes past them, and the first
    # launch holds whole waves of whole tiles
    accepted = 0
    for planes in range(1, shape.D):
        st = capi.conv3d_fp8_describe_status(shape.N, shape.C, shape.D, shape.H, shape.W, shape.K,
                                             shape.T, shape.R, shape.S, shape.stride, shape.pad,
                                             152, overlap=planes)
        if st != capi.CONV3D_OK:
            assert st == capi.CONV3D_EUNSUPPORTED
            continue
        i = _describe(shape, overlap=planes)
        read_upto, first_written, q_a = _overlap_reads_and_writes(shape, i)
        # the padded planes below first_written are whole after the first pack (positions
        # [0, q_a)); the light pack writes from position q_a on, in plane first_written or later
        assert read_upto < first_written, (planes, read_upto, first_written)
        assert i["overlap_units"] % (i["grid"] // 2) == 0 and i["overlap_units"] <= i["full_tiles"]
        assert q_a % 256 == 0 and q_a < shape.D * shape.H * shape.W
        accepted += 1
    assert accepted > 0


def test_describe_channels_last_input(lib):
    # the TMA routes read the caller's NDHWC x: no copy of x in the workspace; the gather route
    # still keeps its zero-padded copy
    for cfg in (2, 4):
        s = synth.CONFIGS[cfg]
        for r in (2, 3):
            a = _describe(s, route=r, splits=1)
            b = _describe(s, route=r, splits=1, input_layout=1)
            assert a["workspace_bytes"] - b["workspace_bytes"] >= s.N * s.C * s.D * s.H * s.W
        g = _describe(s, route=1, splits=1, cta_pair=1)
        assert _describe(s, route=1, splits=1, cta_pair=1, input_layout=1)["workspace_bytes"] == \
            g["workspace_bytes"]
    # reading a channels-last x, the padded-grid route walks an im2col box: pads up to 15 only
    assert _describe(synth.ConvShape(1, 32, 4, 4, 4, 16, pad=16), input_layout=1)["route"] == 2
    assert _describe(synth.ConvShape(1, 32, 4, 4, 4, 16, pad=17), input_layout=1)["route"] == 1
    assert capi.conv3d_fp8_describe_status(1, 32, 4, 4, 4, 16, 3, 3, 3, 1, 16, 152, route=3,
                                           input_layout=1) == capi.CONV3D_EUNSUPPORTED
    assert _describe(synth.ConvShape(1, 32, 4, 4, 4, 16, pad=16))["route"] == 3
    assert capi.conv3d_fp8_describe_status(1, 32, 4, 4, 4, 16, 3, 3, 3, 1, 1, 152,
                                           input_layout=2) == capi.CONV3D_EINVAL


def test_describe_bf16_twin(lib):
    d = lambda s, **kw: capi.conv3d_bf16_describe(s.N, s.C, s.D, s.H, s.W, s.K, s.T, s.R, s.S,
                                                  s.stride, s.pad, 152, **kw)
    for cfg, s in enumerate(synth.CONFIGS):
        a, b = _describe(s), d(s)
        assert b["k_gemm"] == a["k_gemm"] == s.C * s.T * s.R * s.S   # elements
        assert b["route"] == a["route"] and b["cta_pair"] == a["cta_pair"]
        # K blocks are 128 bytes of K_gemm (or, on the padded-grid route, one channel block of a
        # (t, r) pair): the same bytes hold half as many bfloat16 channels
        if b["route"] == 3:
            assert b["k_blocks"] == s.T * s.R * (2 * s.C) // min(128, 2 * s.C)
        else:
            assert b["k_blocks"] == -(-2 * b["k_gemm"] // 128)
    # C in 16-byte units: 8 bfloat16 channels suffice (gather route), 4 do not
    assert d(synth.ConvShape(1, 8, 8, 8, 8, 8))["route"] == 1
    assert capi.conv3d_bf16_describe_status(1, 4, 4, 4, 4, 16, 3, 3, 3, 1, 1,
                                            152) == capi.CONV3D_EUNSUPPORTED
    # 16 channels = 32 bytes: the TMA routes apply
    assert d(synth.ConvShape(1, 16, 8, 8, 8, 16))["route"] in (2, 3)
    # the direct route's explicit im2col holds two-byte elements in the same KCTRS order
    assert d(synth.ConvShape(1, 8, 2, 4, 4, 64))["route"] == 4


def test_describe_tma_epilogue(lib):
    s0 = synth.CONFIGS[0]
    assert _describe(s0)["epilogue"] == 1                            # default: explicit stores
    assert _describe(s0, epilogue=2, route=2)["epilogue"] == 2
    # not on the padded-grid route, not with dhw % 8 != 0 (3*5*7 = 105)
    assert capi.conv3d_fp8_describe_status(1, 32, 8, 8, 8, 32, 3, 3, 3, 1, 1, 152, route=3,
                                           epilogue=2) == capi.CONV3D_EUNSUPPORTED
    assert capi.conv3d_fp8_describe_status(1, 32, 3, 5, 7, 32, 3, 3, 3, 1, 1, 152, route=2,
                                           epilogue=2) == capi.CONV3D_EUNSUPPORTED
    assert capi.conv3d_fp8_describe_status(1, 32, 3, 5, 7, 32, 3, 3, 3, 1, 1, 152,
                                           epilogue=3) == capi.CONV3D_EINVAL


def test_describe_forced_options(lib):
    s = synth.CONFIGS[1]
    i = _describe(s, splits=4, block_n=64, max_ctas=10, cta_pair=1)
    assert i["splits"] == 4 and i["block_n"] == 64 and i["n_tiles"] == 2 and i["grid"] == 10
    # more splits than K blocks collapses to one block per split
    i = _describe(s, splits=10_000)
    assert i["splits"] == i["k_blocks"] and i["k_blocks_per_split"] == 1


@pytest.mark.parametrize("args,code", [
    ((0, 16, 4, 4, 4, 16, 3, 3, 3, 1, 1), capi.CONV3D_EINVAL),    # N = 0
    ((1, 16, 1, 4, 4, 16, 3, 3, 3, 1, 0), capi.CONV3D_EINVAL),    # empty output (D < T, pad 0)
    ((1, 16, 4, 4, 4, 16, 3, 3, 3, 0, 1), capi.CONV3D_EINVAL),    # stride 0
    ((1, 16, 4, 4, 4, 16, 3, 3, 3, 1, -1), capi.CONV3D_EINVAL),   # negative pad
    ((1, 24, 4, 4, 4, 16, 3, 3, 3, 1, 1), capi.CONV3D_EUNSUPPORTED),  # C % 16 != 0
    ((1, 16, 4, 4, 4, 0, 3, 3, 3, 1, 1), capi.CONV3D_EINVAL),     # K = 0
    ((1, 16, 4, 4, 4, 16, 0, 3, 3, 1, 1), capi.CONV3D_EINVAL),    # empty filter
    # index ranges beyond 32 bits: npq = 2^31 rows, and 2^40 bytes of y
    ((2048, 16, 1024, 1024, 1, 16, 1, 1, 1, 1, 0), capi.CONV3D_EUNSUPPORTED),
    ((1, 16, 1024, 1024, 1024, 1 << 20, 1, 1, 1, 1, 0), capi.CONV3D_EUNSUPPORTED),
    ((1, 1 << 28, 1, 1, 1, 16, 1, 1, 1, 1, 0), capi.CONV3D_EUNSUPPORTED),  # C * elem overflow guard
])
def test_describe_validation(lib, args, code):
    N, C, D, H, W, K, T, R, S, st, pd = args
    assert capi.conv3d_fp8_describe_status(N, C, D, H, W, K, T, R, S, st, pd, 152) == code


def test_describe_rejects_bad_block_n(lib):
    s = synth.CONFIGS[0]
    for bn in (16, 48, 288):
        assert capi.conv3d_fp8_describe_status(s.N, s.C, s.D, s.H, s.W, s.K, 3, 3, 3, 1, 1, 152,
                                               block_n=bn) == capi.CONV3D_EINVAL


def test_plan_rejects_bad_shape_before_touching_a_device(lib):
    with pytest.raises(capi.Conv3dFp8Error) as e:
        capi.conv3d_fp8_plan(1, 24, 4, 4, 4, 16, 3, 3, 3, 1, 1)
    assert e.value.status == capi.CONV3D_EUNSUPPORTED


def test_null_plan_entry_points(lib):
    assert capi.conv3d_fp8_workspace_size(None) == 0
    assert lib.conv3d_fp8_check(None) == capi.CONV3D_EINVAL
    capi.conv3d_fp8_destroy(None)
    assert lib.conv3d_fp8_set_timing_events(None, None, None) == capi.CONV3D_EINVAL
    assert lib.conv3d_fp8_set_pack_timing_event(None, None) == capi.CONV3D_EINVAL
    # the host-buffer runs reject a missing plan before any copy or allocation
    st3 = (ctypes.c_int * 3)(1, 1, 1)
    assert lib.conv3d_fp8_run_host(None, None, None, None, None, st3, st3,
                                   None) == capi.CONV3D_EINVAL
    assert lib.conv3d_bf16_run_host(None, None, None, None, st3, st3, None) == capi.CONV3D_EINVAL
