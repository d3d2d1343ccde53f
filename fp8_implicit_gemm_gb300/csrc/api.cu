// api.cu -- the C ABI declared in include/conv3d_fp8.h: planning, validation and launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>

#include "conv3d_fp8.h"
#include "conv3d_fp8_internal.h"

using namespace c3d;

struct conv3d_fp8_plan_s {
  int device = -1;
  int stride[3] = {0, 0, 0};
  int pad[3] = {0, 0, 0};
  ConvParams p{};
  CUtensorMap wmap{};
  CUtensorMap xmap{};  // A tensor map (TMA routes)
  const void* xmap_src = nullptr;  // caller's x the A map was last encoded for (channels-last x)
  CUtensorMap ymap{};              // y as [N][K][dhw] bf16 (TMA-store epilogue)
  const void* ymap_src = nullptr;  // caller's y the map was last encoded for
  const void* wmap_src = nullptr;  // caller's w the B map was last encoded for (direct route)
  int elem_bytes = 1;              // 1: e4m3 plan (conv3d_fp8_*), 2: bfloat16 plan (conv3d_bf16_*)
  const float* ones = nullptr;     // device fp32 {1, 1}: the scales of a bfloat16 plan's runs
  conv3d_fp8_plan_info info{};
  void* workspace = nullptr;
  cudaEvent_t ev_begin = nullptr;  // measurement hook, caller-owned
  cudaEvent_t ev_end = nullptr;
  cudaEvent_t ev_pack = nullptr;   // measurement hook before the pack, caller-owned
  void* host_stage = nullptr;      // device copies of the host-buffer runs' x, w, scales and y
};

namespace {

constexpr unsigned long long kDefaultTimeoutNs = 2000ull * 1000ull * 1000ull;

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }
long long round_up(long long a, long long b) { return ceil_div(a, b) * b; }

int out_dim(int in, int k, int stride, int pad) {
  const long long span = (long long)in + 2LL * pad - k;
  if (stride <= 0 || span < 0) return 0;
  return (int)(span / stride + 1);
}

int next_pow2(int v) {
  int r = 1;
  while (r < v) r <<= 1;
  return r;
}

// Whether some tiles are split along K (their fp32 partials then need the reduction kernel).
bool has_split_tiles(const ConvParams& p) {
  return p.full_tiles < (long long)p.m_tiles * p.n_tiles;
}

struct Layout {
  size_t xp_off, xp_bytes, wp_off, wp_bytes, part_off, part_bytes, status_off, total;
};

// Validation and every tiling decision, with no device access. `pair_slots` > 0 caps the number
// of CTA pairs that can be resident at once (the device's cluster occupancy), when known.
conv3d_status decide(int elem_bytes, int N, int C, int D, int H, int W, int K, int T, int R, int S,
                     const int stride[3], const int pad[3], int sm_count,
                     const conv3d_fp8_options* opts, conv3d_fp8_plan_info* info, ConvParams* pp,
                     Layout* lay, int pair_slots = 0) {
  if (!stride || !pad || !info) return CONV3D_EINVAL;
  if (N <= 0 || C <= 0 || D <= 0 || H <= 0 || W <= 0 || K <= 0 || T <= 0 || R <= 0 || S <= 0)
    return CONV3D_EINVAL;
  for (int i = 0; i < 3; ++i)
    if (stride[i] <= 0 || pad[i] < 0) return CONV3D_EINVAL;
  if (sm_count <= 0) return CONV3D_EINVAL;
  const int Do = out_dim(D, T, stride[0], pad[0]);
  const int Ho = out_dim(H, R, stride[1], pad[1]);
  const int Wo = out_dim(W, S, stride[2], pad[2]);
  if (Do <= 0 || Ho <= 0 || Wo <= 0) return CONV3D_EINVAL;
  if (elem_bytes != 1 && elem_bytes != 2) return CONV3D_EINVAL;
  if (C >= (1 << 28)) return CONV3D_EUNSUPPORTED;
  // From here on C counts the BYTES of one pixel's channels: every tile, stage, descriptor and
  // tensor map below is laid out in bytes, the same for e4m3 and bfloat16 inputs.
  const int C_el = C;
  C *= elem_bytes;
  if (C % 16 != 0) return CONV3D_EUNSUPPORTED;

  const long long dhw = (long long)Do * Ho * Wo;
  const long long npq = (long long)N * dhw;
  const long long taps = (long long)T * R * S;
  const long long kg = taps * C;
  conv3d_fp8_options o{};
  if (opts) o = *opts;
  if (o.route < 0 || o.route > 4 || o.cta_pair < 0 || o.cta_pair > 2 || o.input_layout < 0 ||
      o.input_layout > 1 || o.epilogue < 0 || o.epilogue > 2)
    return CONV3D_EINVAL;
  const bool x_cl = o.input_layout == 1;  // the caller's x is channels-last
  // The TMA im2col route needs C in whole 32-byte sub-tile rows and bounding-box corners
  // (-pad, pad - (filter - 1)) inside the [-16, 15] range of a rank-5 im2col tensor map.
  bool im2col_ok = (C % 32 == 0);
  const int filt[3] = {T, R, S};
  for (int i = 0; i < 3; ++i) {
    const int lower = -pad[i], upper = pad[i] - (filt[i] - 1);
    if (lower < -16 || lower > 15 || upper < -16 || upper > 15 || stride[i] > 8) im2col_ok = false;
  }
  if (o.route == 2 && !im2col_ok) return CONV3D_EUNSUPPORTED;
  // The padded-grid route (CTA pairs only) needs stride 1 on every axis, whole 32-byte channel
  // blocks and an A tile of 128 + S - 1 <= 256 rows; reading a channels-last x of the caller it
  // also needs pads up to 15 (its im2col bounding box runs from -pad to extent - 1 + pad). By
  // default it is taken when the rows of the padded grid that are not outputs cost at most 30%
  // extra MMA work.
  const bool grid_ok = C % 32 == 0 && stride[0] == 1 && stride[1] == 1 && stride[2] == 1 &&
                       S <= 129 && o.cta_pair != 1 &&
                       (!x_cl || (pad[0] <= 15 && pad[1] <= 15 && pad[2] <= 15));
  if (o.route == 3 && !grid_ok) return CONV3D_EUNSUPPORTED;
  // The direct route (one CTA) leaves the weights as the caller holds them: B is read by TMA
  // tiles of the KCTRS weights viewed as [K][C*T*R*S] (rows of a multiple of 16 bytes), and the
  // pre-pass writes A = im2col(x) explicitly, [npq][C*T*R*S] in the same (channel, tap) order, for
  // TMA tiles too. By default it is taken for layers with at most four 128-row tiles and no more
  // output positions than output channels, where the explicit A (npq rows) is smaller than the
  // weights (K rows) that the other routes re-lay every run.
  const long long x_bytes_in = (long long)N * C * D * H * W;
  const bool direct_ok = !x_cl && kg % 16 == 0 && x_bytes_in < (1LL << 31) && o.cta_pair != 2;
  if (o.route == 4 && !direct_ok) return CONV3D_EUNSUPPORTED;
  const double grid_overhead =
      (double)(H + 2LL * pad[1]) * (double)(W + 2LL * pad[2]) / ((double)Ho * (double)Wo);
  int route;
  if (o.route == 1)
    route = kRouteGather;
  else if (o.route == 2)
    route = kRouteIm2col;
  else if (o.route == 3)
    route = kRouteGrid;
  else if (o.route == 4)
    route = kRouteDirect;
  else if (grid_ok && grid_overhead <= 1.3 && npq > kBlockM)
    route = kRouteGrid;
  else if (direct_ok && npq <= 4LL * kBlockM && npq <= K)
    route = kRouteDirect;
  else
    route = im2col_ok ? kRouteIm2col : kRouteGather;
  const int a_cb = C % 128 == 0 ? 128 : (C % 64 == 0 ? 64 : 32);
  // TMA-store epilogue: the output-position routes (a tile's rows are consecutive positions of
  // one image's dhw run), with dhw a multiple of 8 (16-byte rows of the map of y and 16-byte
  // aligned box starts). By default the explicit guarded stores.
  const bool epi_ok = route != kRouteGrid && dhw % 8 == 0;
  if (o.epilogue == 2 && !epi_ok) return CONV3D_EUNSUPPORTED;
  const bool epi_tma = o.epilogue == 2;
  // A zero-padded channels-last copy of x for the gather route, and for the padded-grid route
  // when the library transposes x anyway; the TMA routes read a channels-last x of the caller
  // directly (no copy at all), and the im2col route's copy needs no halo.
  const bool direct = route == kRouteDirect;
  const bool keep_copy = (!x_cl || route == kRouteGather) && !direct;
  const bool halo_on = route == kRouteGather || (route == kRouteGrid && !x_cl);
  const int halo[3] = {halo_on ? pad[0] : 0, halo_on ? pad[1] : 0, halo_on ? pad[2] : 0};
  const long long Dp = D + 2LL * halo[0], Hp = H + 2LL * halo[1], Wp = W + 2LL * halo[2];
  const long long Dg = D + 2LL * pad[0], Hg = H + 2LL * pad[1], Wg = W + 2LL * pad[2];
  const long long y_elems = npq * K;
  const long long x_elems = (long long)N * C * D * H * W;
  // the direct route's buffer is the explicit A = im2col(x), npq rows of kg bytes
  const long long xp_elems = keep_copy ? (long long)N * Dp * Hp * Wp * C : (direct ? npq * kg : 0);
  // 32-bit limits of the index arithmetic inside the kernels.
  if (npq + kBlockM >= (1LL << 31) || kg + kBlockK >= (1LL << 31) || y_elems >= (1LL << 40) ||
      x_elems >= (1LL << 40) || xp_elems >= (1LL << 40) || Dg >= (1LL << 30) ||
      Hg >= (1LL << 30) || Wg >= (1LL << 30) || K >= (1 << 30) || taps >= (1 << 20))
    return CONV3D_EUNSUPPORTED;

  int block_n = o.block_n;
  if (block_n == 0) block_n = (int)std::min<long long>(256, round_up(K, 32));
  if (block_n < 32 || block_n > 256 || block_n % 32 != 0) return CONV3D_EINVAL;

  // CTA pairs (cta_group::2, 256-row tiles) run the im2col and padded-grid routes. The im2col
  // route runs on one CTA unless asked: on every shape measured the one-CTA kernel was faster
  // there (N tile 64-256, 4-10%: e.g. 313.6 against 342.2 us on the large layer, 61.9 against
  // 68.2 us on a stride-2 layer of the vae shape).
  if (o.cta_pair == 2 && route == kRouteGather) return CONV3D_EUNSUPPORTED;
  if (o.cta_pair == 2 && direct) return CONV3D_EUNSUPPORTED;
  const bool pair = route == kRouteGrid || (route == kRouteIm2col && o.cta_pair == 2);
  const int block_m = pair ? 2 * kBlockM : kBlockM;
  // co-resident units: one per SM, or one per CTA pair; a CTA cap given in the options counts
  long long slots = pair ? std::max(1, sm_count / 2) : sm_count;
  if (pair && pair_slots > 0) slots = std::min<long long>(slots, pair_slots);
  if (o.max_ctas > 0)
    slots = std::min<long long>(slots, pair ? std::max(1, o.max_ctas / 2) : o.max_ctas);

  // grid route: the tiles of one image cover the first Do planes of its padded grid
  const long long tiles_per_image =
      route == kRouteGrid ? ceil_div((long long)Do * Hg * Wg, block_m) : 0;
  const long long m_tiles = route == kRouteGrid ? N * tiles_per_image : ceil_div(npq, block_m);
  const long long n_tiles = ceil_div(K, block_n);
  // K blocks: 128 bytes of K_gemm, or on the grid route one (t, r, channel block) group of S taps
  const long long k_blocks =
      route == kRouteGrid ? (long long)T * R * (C / a_cb) : ceil_div(kg, kBlockK);
  if (route == kRouteGrid && (long long)N * Dg * Hg * Wg + 256 >= (1LL << 31))
    return CONV3D_EUNSUPPORTED;
  const long long tiles = m_tiles * n_tiles;
  long long splits = o.splits;
  if (splits < 0) return CONV3D_EINVAL;
  // Tiles 0..full_tiles-1 are computed whole; the rest are split along K. By default: with at most
  // a quarter as many tiles as slots, every tile is split to fill the machine, down to four K
  // blocks a split, or three when the whole K loop is short (under 32 blocks) (with more tiles
  // the reduction of the partials costs more than the shorter K loops save; measured: the p1
  // layer, 21 K blocks, 15.4 us a step in 7 splits against 16.7 in 5; the deep layer, 108
  // blocks, 36 splits of 3 tie 27 of 4, and 54 of 2 lose, 25.5 against 21.5 us; its bfloat16
  // twin, 216 blocks, 27.7 us in 72 splits of 3 against 26.8 in 54 of 4); with more tiles
  // than slots, only the tiles of a last, mostly idle wave are split, over the slots that wave
  // would leave idle, and only when a tile's main loop is long enough (at least 16384 tensor-core
  // cycles: about 8 us) for the shorter tail to repay the reduction's launch and partial traffic
  // (measured: 2 x 64 x 16 x 64 x 64 -> 128, 546 tiles whose K loop is ~3500 cycles: 40.7 us
  // unsplit against 47.4 us with its 14-tile tail split 5 ways; the large layer and a stride-2
  // layer, ~27600 cycles a tile, gain ~6%). A split count in the options splits every tile that
  // many ways.
  // tensor-core cycles of one tile's K loop: MMAs of K = 32 bytes, N / 2 cycles each (M = 128
  // rows per CTA; the padded-grid route issues S taps x a_cb / 32 of them per K block)
  const long long mmas_per_kb = route == kRouteGrid ? (long long)S * (a_cb / 32) : kBlockK / 32;
  const long long tile_cycles = k_blocks * mmas_per_kb * (block_n / 2);
  long long full_tiles = 0;
  if (splits == 0) {
    splits = 1;
    if (tiles * 4 <= slots && k_blocks >= 8) {
      const long long min_kb = k_blocks < 32 ? 3 : 4;
      splits = std::max<long long>(1, std::min<long long>(slots / tiles, k_blocks / min_kb));
    } else if (tiles > slots && k_blocks >= 4 && tile_cycles >= 16384) {
      const long long tail = tiles % slots;
      if (tail > 0 && tail * 2 <= slots) {
        full_tiles = tiles - tail;
        splits = std::min<long long>(slots / tail, k_blocks);
      }
    }
  }
  splits = std::min(splits, k_blocks);
  const long long kbps = ceil_div(k_blocks, splits);
  splits = ceil_div(k_blocks, kbps);  // every split owns at least one K block
  if (splits == 1) full_tiles = tiles;
  const long long units = full_tiles + (tiles - full_tiles) * splits;
  if (units >= (1LL << 31)) return CONV3D_EUNSUPPORTED;

  long long stage_bytes = kATileBytes + (long long)(pair ? block_n / 2 : block_n) * kBlockK;
  if (route == kRouteGrid)
    stage_bytes = round_up((long long)(kBlockM + S - 1) * a_cb, 1024) +
                  round_up((long long)S * (block_n / 2) * a_cb, 1024);
  const int stages = (int)std::min<long long>(kMaxStages, kSmemBudget / stage_bytes);
  if (stages < (route == kRouteGrid ? 2 : 3)) return CONV3D_EUNSUPPORTED;
  long long grid = std::min<long long>(units, slots);
  if (pair) grid *= 2;  // two CTAs per unit
  if (o.max_ctas < 0 || o.wait_timeout_ms < 0 || o.overlap < -1) return CONV3D_EINVAL;

  // Pack beside the GEMM (padded-grid route, one image, an NCDHW x taken by the tiled transpose):
  // the first P input planes are packed before the GEMM starts on the tiles that read only those
  // (whole waves), while a light pack (one block an SM, one 16 KB stage) copies the rest beside
  // it; the remaining units run as a second launch. The pack block must fit beside a GEMM CTA:
  // its shared memory in the SM's 228 KB (1 KB reserved a block), its 256 x 64 registers beside
  // the GEMM's 320 x 128. Measured: a 64 MB copy that takes 45.7 us alone added 7.3 us to the
  // large layer's run when it ran beside the GEMM on one block an SM.
  long long ov_planes = 0, ov_units = 0;
  {
    const long long dhw_in = (long long)D * H * W;
    const long long gemm_smem =
        1024 + stages * stage_bytes + (2LL * stages + 5) * 8 + 16;  // the pair kernel's
    const bool ov_ok = route == kRouteGrid && !x_cl && N == 1 && W % 4 == 0 &&
                       (dhw_in * elem_bytes) % 16 == 0 && C_el % 64 == 0 &&
                       dhw_in < (1LL << 31) && D >= 2 &&
                       gemm_smem + 1024 + kPackLightSmem + 1024 <= kSmemPerSm;
    const long long waves = full_tiles / slots;  // whole waves of whole tiles (a unit each)
    if (o.overlap > 0 && !ov_ok) return CONV3D_EUNSUPPORTED;
    if (ov_ok && (o.overlap > 0 || (o.overlap == 0 && waves >= 4))) {
      // m tiles that read only the padded planes [0, pd + P): the last grid row of tile m plus
      // the farthest tap lies below (pd + P) planes of the padded grid
      const long long reach = (T - 1LL) * Hg * Wg + (R - 1LL) * Wg + (S - 1LL);
      auto units_for = [&](long long P) {
        const long long room = (pad[0] + P) * Hg * Wg - reach;
        const long long m_ok = room > 0 ? room / block_m : 0;
        const long long u = std::min(m_ok * n_tiles, full_tiles);
        return (u / slots) * slots;  // whole waves
      };
      // By default, a cost model of measured rates: a wave of units takes about 1.13 x a tile's
      // tensor-core cycles at 1.9 GHz (the large layer's kernel); the light pack moves about
      // 2.5 TB/s of x beside the GEMM, the whole pack about 6 TB/s alone; the overlap costs
      // about 8 us (the second launch's start, the light pack's pull on the GEMM). P is the
      // fewest planes whose first launch outlasts the light pack of the rest by 10%, taken only
      // when the pack time it saves exceeds that cost (the large layer: P = 5, 3 of 13 waves
      // first; measured best of 4, 5 and 6; the vae layer, 3 waves, measured slower with it).
      const double x_tr_bytes = 2.0 * (double)N * C * dhw_in;  // x read and its copy written
      auto rest_frac = [&](long long P) {
        return (double)(dhw_in - std::min(dhw_in, round_up(P * H * W, kPackTilePositions))) /
               (double)dhw_in;
      };
      long long P = o.overlap > 0 ? o.overlap : 0;
      if (P == 0) {
        for (long long c = 1; c < D && P == 0; ++c) {
          const long long ua = units_for(c);
          if (ua < slots) continue;
          const double t_first_us = (double)(ua / slots) * (double)tile_cycles * 1.13 / 1900.0;
          const double t_light_us = x_tr_bytes * rest_frac(c) / 2.5e6;
          if (t_first_us >= 1.1 * t_light_us) P = c;
        }
        if (P > 0 && x_tr_bytes * rest_frac(P) / 6.0e6 < 8.0) P = 0;  // not worth its cost
      }
      if (P > 0 && P < D && units_for(P) >= slots &&
          round_up(P * H * W, kPackTilePositions) < dhw_in) {
        ov_planes = P;
        ov_units = units_for(P);
      } else if (o.overlap > 0) {
        return CONV3D_EUNSUPPORTED;
      }
    }
  }

  Layout L{};
  L.xp_off = 0;
  L.xp_bytes = (size_t)xp_elems;
  L.wp_off = (size_t)round_up((long long)L.xp_off + L.xp_bytes, 256);
  L.wp_bytes = direct ? 0 : (size_t)(K * kg);  // the direct route reads the caller's weights
  L.part_off = (size_t)round_up((long long)L.wp_off + L.wp_bytes, 256);
  L.part_bytes = (size_t)((tiles - full_tiles) * splits * block_n * block_m * 4);
  L.status_off = (size_t)round_up((long long)L.part_off + L.part_bytes, 256);
  L.total = L.status_off + 256;

  std::memset(info, 0, sizeof(*info));
  info->Do = Do;
  info->Ho = Ho;
  info->Wo = Wo;
  info->npq = npq;
  info->k_gemm = (int)(taps * C_el);
  info->block_m = block_m;
  info->block_n = block_n;
  info->m_tiles = (int)m_tiles;
  info->n_tiles = (int)n_tiles;
  info->k_blocks = (int)k_blocks;
  info->splits = (int)splits;
  info->k_blocks_per_split = (int)kbps;
  info->full_tiles = (int)full_tiles;
  info->epilogue = epi_tma ? 2 : 1;
  info->overlap_planes = (int)ov_planes;
  info->overlap_units = (int)ov_units;
  info->stages = stages;
  info->row_chk = route == kRouteGrid ? 1 : (npq % block_m) != 0;
  info->grid = (int)grid;
  info->sm_count = sm_count;
  info->workspace_bytes = L.total;
  info->route = route == kRouteGrid ? 3 : route == kRouteIm2col ? 2 : route == kRouteDirect ? 4 : 1;
  info->cta_pair = pair ? 2 : 1;

  if (pp) {
    ConvParams& p = *pp;
    std::memset(&p, 0, sizeof(p));
    p.N = N; p.C = C; p.D = D; p.H = H; p.W = W; p.K = K; p.T = T; p.R = R; p.S = S;
    p.elem_bytes = elem_bytes;
    p.sd = stride[0]; p.sh = stride[1]; p.sw = stride[2];
    p.pd = pad[0]; p.ph = pad[1]; p.pw = pad[2];
    p.Do = Do; p.Ho = Ho; p.Wo = Wo;
    p.route = route;
    p.a_cb = a_cb;
    p.pk_pd = halo[0]; p.pk_ph = halo[1]; p.pk_pw = halo[2];
    p.Dp = (int)Dp; p.Hp = (int)Hp; p.Wp = (int)Wp;
    p.Dg = (int)Dg; p.Hg = (int)Hg; p.Wg = (int)Wg;
    p.x_cl = x_cl ? 1 : 0;
    p.epi_tma = epi_tma ? 1 : 0;
    p.halo_once = 1;  // a plan zeroes its padded copy once (the allocation-free entry does not)
    p.a_grid_im2col = route == kRouteGrid && x_cl ? 1 : 0;
    p.dhw = (int)dhw;
    p.tiles_per_image = (int)tiles_per_image;
    p.npq = (int)npq;
    p.taps = (int)taps;
    p.kg = (int)kg;
    p.pair = pair ? 1 : 0;
    p.block_m = block_m;
    p.block_n = block_n;
    p.m_tiles = (int)m_tiles;
    p.n_tiles = (int)n_tiles;
    p.k_blocks = (int)k_blocks;
    p.splits = (int)splits;
    p.kb_per_split = (int)kbps;
    p.full_tiles = (int)full_tiles;
    p.num_units = (int)units;
    p.stages = stages;
    p.acc_stride = std::max(32, next_pow2(block_n));
    p.tmem_cols = 2 * p.acc_stride;
    p.timeout_ns = o.wait_timeout_ms > 0 ? (unsigned long long)o.wait_timeout_ms * 1000000ull
                                         : kDefaultTimeoutNs;
    p.debug_flags = o.debug_flags;
  }
  if (lay) *lay = L;
  return CONV3D_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

CUtensorMapSwizzle swizzle_for(int row_bytes) {
  return row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
         : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                           : CU_TENSOR_MAP_SWIZZLE_32B;
}

// A 2D byte tensor [rows][cols] (row pitch = cols); a box is box_cols bytes of box_rows rows,
// written to shared memory with the swizzle of its row width.
conv3d_status encode_2d(CUtensorMap* map, void* base, long long rows, long long cols, int box_cols,
                        int box_rows) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return CONV3D_ECUDA;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(box_cols),
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV3D_OK : CONV3D_ECUDA;
}

typedef CUresult (*EncodeIm2colFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const int*, const int*,
                                   cuuint32_t, cuuint32_t, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeIm2colFn get_encode_im2col() {
  static EncodeIm2colFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeIm2colFn>(ptr);
  }
  return fn;
}

// The packed x as a channels-last 5D tensor (C, W, H, D, N), read in im2col mode; everything
// outside the tensor reads zero. im2col route: one load brings 128 consecutive output positions
// (the traversal walks W, then H, D and N, over the starting pixels of the filter windows: from
// -pad to extent - 1 + pad - (filter - 1), every `stride`), a_cb channels each, shifted by the
// tap given with the load. Padded-grid route: the traversal walks the whole zero-padded grid
// (from -pad to extent - 1 + pad, stride 1) and one load brings 128 + S - 1 consecutive grid
// positions, shifted by the (r, t) of the load; the S taps along W are row offsets into it.
conv3d_status encode_im2col_map(CUtensorMap* map, void* xcl, const ConvParams& p, bool grid) {
  EncodeIm2colFn enc = get_encode_im2col();
  if (!enc) return CONV3D_ECUDA;
  const cuuint64_t dims[5] = {(cuuint64_t)p.C, (cuuint64_t)p.W, (cuuint64_t)p.H, (cuuint64_t)p.D,
                              (cuuint64_t)p.N};
  const cuuint64_t strides[4] = {(cuuint64_t)p.C, (cuuint64_t)p.C * p.W,
                                 (cuuint64_t)p.C * p.W * p.H, (cuuint64_t)p.C * p.W * p.H * p.D};
  const int lower[3] = {-p.pw, -p.ph, -p.pd};
  int upper[3] = {p.pw - (p.S - 1), p.ph - (p.R - 1), p.pd - (p.T - 1)};
  if (grid) {
    upper[0] = p.pw;
    upper[1] = p.ph;
    upper[2] = p.pd;
  }
  const cuuint32_t rows = grid ? (cuuint32_t)(kBlockM + p.S - 1) : (cuuint32_t)kBlockM;
  const cuuint32_t estr[5] = {1, (cuuint32_t)p.sw, (cuuint32_t)p.sh, (cuuint32_t)p.sd, 1};
  const CUtensorMapSwizzle sw = p.a_cb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : p.a_cb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, xcl, dims, strides, lower, upper,
                   (cuuint32_t)p.a_cb, rows, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV3D_OK : CONV3D_ECUDA;
}

// y as a bf16 tensor [N][K][dhw] (dhw innermost) for the TMA-store epilogue: a box is 128
// positions of 32 channels of one image; stores outside the extents are dropped by the TMA unit.
conv3d_status encode_ymap(CUtensorMap* map, const ConvParams& p, void* y) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return CONV3D_ECUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)p.dhw, (cuuint64_t)p.K, (cuuint64_t)p.N};
  const cuuint64_t strides[2] = {(cuuint64_t)p.dhw * 2, (cuuint64_t)p.K * p.dhw * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kBlockM, 32u, 1u};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, y, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CONV3D_OK : CONV3D_ECUDA;
}

// Whether the A tensor map reads the caller's x (a channels-last x on a TMA route), so that it is
// encoded per run rather than once per plan.
bool xmap_reads_caller_x(const ConvParams& p) { return p.x_cl && p.route != kRouteGather; }

// A tensor map of a plan: im2col map of the unpadded channels-last x (the im2col route, and the
// padded-grid route reading a channels-last x of the caller), or 2D tiles of 128 + S - 1 rows of
// the zero-padded copy viewed as [N*Dg*Hg*Wg][C] (padded-grid route). `x_cl` is the caller's
// channels-last x, used when the map reads it.
conv3d_status encode_xmap(CUtensorMap* xmap, const ConvParams& p, const void* x_cl) {
  void* src = xmap_reads_caller_x(p) ? const_cast<void*>(x_cl) : static_cast<void*>(p.xp);
  if (p.route == kRouteIm2col) return encode_im2col_map(xmap, src, p, false);
  if (p.route == kRouteGrid) {
    if (p.a_grid_im2col) return encode_im2col_map(xmap, src, p, true);
    return encode_2d(xmap, src, (long long)p.N * p.Dg * p.Hg * p.Wg, p.C, p.a_cb,
                     kBlockM + p.S - 1);
  }
  // direct route: 128-row tiles of one 128-byte K block of the explicit A = im2col(x)
  if (p.route == kRouteDirect) return encode_2d(xmap, src, p.npq, p.kg, kBlockK, kBlockM);
  return CONV3D_OK;
}

// B tensor map: weights viewed as [K][kg] bytes (the packed K x taps x C copy, or on the direct
// route the caller's KCTRS w, whose rows hold the same kg bytes in channel-outer order); a box is
// one K block (128 bytes, or a_cb bytes of one tap on the grid route) of block_n rows
// (block_n / 2 per CTA of a pair).
conv3d_status encode_wmap(CUtensorMap* wmap, const ConvParams& p, const void* w) {
  const int b_rows = p.pair ? p.block_n / 2 : p.block_n;
  const int b_cols = p.route == kRouteGrid ? p.a_cb : kBlockK;
  return encode_2d(wmap, const_cast<void*>(w), p.K, p.kg, b_cols, b_rows);
}

// Tensor maps of a plan: B over the packed weights (the direct route encodes it per run, over the
// caller's w); A as above, unless it reads the caller's x (then each run encodes it).
conv3d_status encode_maps(CUtensorMap* wmap, CUtensorMap* xmap, const ConvParams& p) {
  if (p.route != kRouteDirect) {
    const conv3d_status st = encode_wmap(wmap, p, p.wp);
    if (st != CONV3D_OK) return st;
  }
  if (xmap_reads_caller_x(p)) return CONV3D_OK;
  return encode_xmap(xmap, p, nullptr);
}

struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  cudaError_t set(int dev) {
    cudaError_t e = cudaGetDevice(&prev);
    if (e != cudaSuccess) return e;
    if (prev != dev) {
      e = cudaSetDevice(dev);
      changed = (e == cudaSuccess);
    }
    return e;
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

conv3d_status conv3d_fp8_describe(int N, int C, int D, int H, int W, int K, int T, int R, int S,
                                  const int stride[3], const int pad[3], int sm_count,
                                  const conv3d_fp8_options* opts, conv3d_fp8_plan_info* info) {
  return decide(1, N, C, D, H, W, K, T, R, S, stride, pad, sm_count, opts, info, nullptr, nullptr);
}

}  // extern "C"

namespace {

// Plans of both input types: e4m3 (elem_bytes 1) and bfloat16 (elem_bytes 2).
conv3d_status plan_impl(int elem_bytes, conv3d_fp8_plan_t* out, int N, int C, int D, int H, int W,
                        int K, int T, int R, int S, const int stride[3], const int pad[3],
                        int device, const conv3d_fp8_options* opts) {
  if (!out) return CONV3D_EINVAL;
  *out = nullptr;
  // Shape errors first, without touching any device.
  conv3d_fp8_plan_info probe{};
  conv3d_status st = decide(elem_bytes, N, C, D, H, W, K, T, R, S, stride, pad, 1, opts, &probe,
                            nullptr, nullptr);
  if (st != CONV3D_OK) return st;

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev <= 0) {
    cudaGetLastError();
    return CONV3D_ECUDA;
  }
  if (device < 0 || device >= ndev) return CONV3D_EINVAL;
  DeviceGuard guard;
  if (guard.set(device) != cudaSuccess) return CONV3D_ECUDA;
  cudaDeviceProp prop{};
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return CONV3D_ECUDA;
  if (prop.major != 10 || prop.minor != 3) return CONV3D_EUNSUPPORTED;

  conv3d_fp8_plan_s* plan = new (std::nothrow) conv3d_fp8_plan_s();
  if (!plan) return CONV3D_ENOMEM;
  Layout L{};
  st = decide(elem_bytes, N, C, D, H, W, K, T, R, S, stride, pad, prop.multiProcessorCount, opts,
              &plan->info, &plan->p, &L);
  if (st != CONV3D_OK) {
    delete plan;
    return st;
  }
  // The attribute is per kernel and per device, shared by every plan: grant the device's opt-in
  // maximum once, so that a later plan with a smaller tile cannot shrink it under this one. It
  // comes before the occupancy query below, which counts clusters at this plan's shared memory.
  if (conv_set_smem_attr((size_t)prop.sharedMemPerBlockOptin) != cudaSuccess) {
    delete plan;
    return CONV3D_ECUDA;
  }
  if (plan->p.pair) {  // plan for the CTA pairs the device can actually hold at once
    const int clusters = conv_pair_max_active_clusters(plan->p);
    if (clusters > 0 && clusters < prop.multiProcessorCount / 2) {
      st = decide(elem_bytes, N, C, D, H, W, K, T, R, S, stride, pad, prop.multiProcessorCount,
                  opts, &plan->info, &plan->p, &L, clusters);
      if (st != CONV3D_OK) {
        delete plan;
        return st;
      }
    }
  }
  plan->device = device;
  for (int i = 0; i < 3; ++i) {
    plan->stride[i] = stride[i];
    plan->pad[i] = pad[i];
  }
  const size_t smem = plan->p.pair
                         ? conv_pair_smem_bytes(plan->p)
                         : conv_smem_bytes(plan->p.block_n, plan->p.stages, plan->p.epi_tma != 0);
  if ((int)smem > prop.sharedMemPerBlockOptin) {
    delete plan;
    return CONV3D_EUNSUPPORTED;
  }
  if (cudaMalloc(&plan->workspace, L.total) != cudaSuccess) {
    cudaGetLastError();
    delete plan;
    return CONV3D_ENOMEM;
  }
  uint8_t* ws = static_cast<uint8_t*>(plan->workspace);
  plan->p.xp = L.xp_bytes ? ws + L.xp_off : nullptr;
  plan->p.wp = ws + L.wp_off;
  plan->p.partials = L.part_bytes ? reinterpret_cast<float*>(ws + L.part_off) : nullptr;
  plan->p.status = reinterpret_cast<int*>(ws + L.status_off);
  // the zero halo of the padded copy, once: no run writes it again
  if (L.xp_bytes && cudaMemset(plan->p.xp, 0, L.xp_bytes) != cudaSuccess) {
    cudaFree(plan->workspace);
    delete plan;
    return CONV3D_ECUDA;
  }
  // The status word at offset 0 of its 256-byte slot; a bfloat16 plan keeps two fp32 ones at
  // offset 128, the scales its runs pass to the kernels (its inputs carry no scale).
  const float ones[2] = {1.0f, 1.0f};
  if (cudaMemset(plan->p.status, 0, 256) != cudaSuccess ||
      (elem_bytes == 2 && cudaMemcpy(ws + L.status_off + 128, ones, sizeof ones,
                                     cudaMemcpyHostToDevice) != cudaSuccess)) {
    cudaFree(plan->workspace);
    delete plan;
    return CONV3D_ECUDA;
  }
  plan->elem_bytes = elem_bytes;
  plan->ones = reinterpret_cast<const float*>(ws + L.status_off + 128);
  if (plan->p.pair) {  // never more clusters than can be resident at once
    const int clusters = conv_pair_max_active_clusters(plan->p);
    if (clusters > 0 && plan->info.grid > 2 * clusters) plan->info.grid = 2 * clusters;
  }
  st = encode_maps(&plan->wmap, &plan->xmap, plan->p);
  if (st != CONV3D_OK) {
    cudaFree(plan->workspace);
    delete plan;
    return st;
  }
  if (plan->info.overlap_planes > 0 &&
      smem + 1024 + (size_t)kPackLightSmem + 1024 > (size_t)prop.sharedMemPerMultiprocessor) {
    // this device's SM cannot hold a pack block beside a GEMM CTA: the pack runs whole first
    plan->info.overlap_planes = 0;
    plan->info.overlap_units = 0;
  }
  *out = plan;
  return CONV3D_OK;
}

// Runs of both input types; the bfloat16 entry passes the plan's fp32 ones as the scales.
conv3d_status run_impl(conv3d_fp8_plan_t plan, const void* x, const void* w,
                       const float* scale_x, const float* scale_w, void* y,
                       const int stride[3], const int pad[3], void* stream,
                       int x_src_type = kSrcE4m3) {
  if (!plan || !x || !w || !scale_x || !scale_w || !y || !stride || !pad) return CONV3D_EINVAL;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(scale_x, 4) ||
      !aligned(scale_w, 4))
    return CONV3D_EINVAL;
  for (int i = 0; i < 3; ++i)
    if (stride[i] != plan->stride[i] || pad[i] != plan->pad[i]) return CONV3D_EINVAL;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return CONV3D_ECUDA;
  if (cur != plan->device) return CONV3D_EINVAL;

  ConvParams p = plan->p;
  p.x_src_type = x_src_type;
  p.x = static_cast<const uint8_t*>(x);
  p.w = static_cast<const uint8_t*>(w);
  p.y = static_cast<uint16_t*>(y);
  p.scale_x = scale_x;
  p.scale_w = scale_w;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (xmap_reads_caller_x(p) && plan->xmap_src != x) {
    const conv3d_status st = encode_xmap(&plan->xmap, p, x);
    if (st != CONV3D_OK) return st;
    plan->xmap_src = x;
  }
  if (p.epi_tma && plan->ymap_src != y) {
    const conv3d_status st = encode_ymap(&plan->ymap, p, y);
    if (st != CONV3D_OK) return st;
    plan->ymap_src = y;
  }
  const bool direct = p.route == kRouteDirect;  // B is read from the caller's w as it is
  if (direct && plan->wmap_src != w) {
    const conv3d_status st = encode_wmap(&plan->wmap, p, w);
    if (st != CONV3D_OK) return st;
    plan->wmap_src = w;
  }
  if (plan->ev_pack && cudaEventRecord(plan->ev_pack, s) != cudaSuccess) return CONV3D_ECUDA;
  const bool row_chk = plan->info.row_chk != 0;
  if (plan->info.overlap_planes > 0 && x_src_type == kSrcE4m3 && pack_transposes_x(p)) {
    // The pack beside the GEMM, as one chain of programmatic dependent launches on the caller's
    // stream: the first planes of x and the weights; the GEMM on the units that read only those
    // (whole waves); the light pack of the other planes (one block an SM), launched once every
    // CTA of that GEMM has passed its wait on the first pack and triggered its dependents, so
    // that it only takes the room left beside them, and never waiting on that GEMM; the second
    // GEMM launch on the remaining units, whose CTAs take the SMs the first launch frees and
    // whose wait covers the light pack (the first pack completed before it began); the
    // reduction of the split tiles.
    const long long dhw_in = (long long)p.D * p.H * p.W;
    const long long q_a = std::min<long long>(
        dhw_in, round_up((long long)plan->info.overlap_planes * p.H * p.W, kPackTilePositions));
    ConvParams pa = p, pb = p;
    pa.num_units = plan->info.overlap_units;
    pb.unit_base = pa.num_units;
    pb.num_units = p.num_units - pa.num_units;
    const int grid_a = std::min(plan->info.grid, 2 * pa.num_units);
    const int grid_b = std::min(plan->info.grid, 2 * pb.num_units);
    if (launch_pack_range(p, 0, q_a, true, false, s) != cudaSuccess) return CONV3D_ECUDA;
    if (plan->ev_begin && cudaEventRecord(plan->ev_begin, s) != cudaSuccess) return CONV3D_ECUDA;
    if (launch_conv(pa, plan->wmap, plan->xmap, plan->ymap, row_chk, grid_a, s) != cudaSuccess ||
        launch_pack_range(p, q_a, dhw_in, false, true, s) != cudaSuccess ||
        launch_conv(pb, plan->wmap, plan->xmap, plan->ymap, row_chk, grid_b, s) != cudaSuccess)
      return CONV3D_ECUDA;
    if (has_split_tiles(p) && launch_splitk_reduce(p, row_chk, s) != cudaSuccess)
      return CONV3D_ECUDA;
  } else {
    if (launch_pack(p, s) != cudaSuccess) return CONV3D_ECUDA;
    if (plan->ev_begin && cudaEventRecord(plan->ev_begin, s) != cudaSuccess) return CONV3D_ECUDA;
    if (launch_conv(p, plan->wmap, plan->xmap, plan->ymap, row_chk, plan->info.grid, s) !=
        cudaSuccess)
      return CONV3D_ECUDA;
    if (has_split_tiles(p) && launch_splitk_reduce(p, row_chk, s) != cudaSuccess)
      return CONV3D_ECUDA;
  }
  if (plan->ev_end && cudaEventRecord(plan->ev_end, s) != cudaSuccess) return CONV3D_ECUDA;
  return CONV3D_OK;
}

// Runs with host buffers: x, w and (e4m3 plans) the two scales are copied into device buffers the
// plan owns, the run reads them there, and y is copied back; one cudaMemcpyAsync per copy, all on
// the caller's stream, in that order.
conv3d_status run_host_impl(conv3d_fp8_plan_t plan, const void* x_host, const void* w_host,
                            const float* scales_host, void* y_host, const int stride[3],
                            const int pad[3], void* stream) {
  if (!plan || !x_host || !w_host || !y_host || !stride || !pad) return CONV3D_EINVAL;
  if (plan->elem_bytes == 1 && !scales_host) return CONV3D_EINVAL;
  for (int i = 0; i < 3; ++i)
    if (stride[i] != plan->stride[i] || pad[i] != plan->pad[i]) return CONV3D_EINVAL;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return CONV3D_ECUDA;
  if (cur != plan->device) return CONV3D_EINVAL;
  const ConvParams& q = plan->p;  // C counts bytes of a pixel
  const size_t x_bytes = (size_t)q.N * q.C * q.D * q.H * q.W;
  const size_t w_bytes = (size_t)q.K * q.C * q.taps;
  const size_t y_bytes = (size_t)q.npq * q.K * 2;
  const size_t off_w = (size_t)round_up((long long)x_bytes, 256);
  const size_t off_s = off_w + (size_t)round_up((long long)w_bytes, 256);
  const size_t off_y = off_s + 256;
  const size_t total = off_y + (size_t)round_up((long long)y_bytes, 256);
  if (!plan->host_stage && cudaMalloc(&plan->host_stage, total) != cudaSuccess) {
    cudaGetLastError();
    plan->host_stage = nullptr;
    return CONV3D_ENOMEM;
  }
  uint8_t* st = static_cast<uint8_t*>(plan->host_stage);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(st, x_host, x_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(st + off_w, w_host, w_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return CONV3D_ECUDA;
  const float* sx = plan->ones;
  const float* sw = plan->ones + 1;
  if (plan->elem_bytes == 1) {
    if (cudaMemcpyAsync(st + off_s, scales_host, 2 * sizeof(float), cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
      return CONV3D_ECUDA;
    sx = reinterpret_cast<const float*>(st + off_s);
    sw = sx + 1;
  }
  const conv3d_status rs = run_impl(plan, st, st + off_w, sx, sw, st + off_y, stride, pad, stream);
  if (rs != CONV3D_OK) return rs;
  if (cudaMemcpyAsync(y_host, st + off_y, y_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CONV3D_ECUDA;
  return CONV3D_OK;
}

}  // namespace

extern "C" {

conv3d_status conv3d_fp8_run_host(conv3d_fp8_plan_t plan, const void* x_host, const void* w_host,
                                  const float* scales, void* y_host, const int stride[3],
                                  const int pad[3], void* stream) {
  if (plan && plan->elem_bytes != 1) return CONV3D_EINVAL;
  return run_host_impl(plan, x_host, w_host, scales, y_host, stride, pad, stream);
}

conv3d_status conv3d_bf16_run_host(conv3d_fp8_plan_t plan, const void* x_host, const void* w_host,
                                   void* y_host, const int stride[3], const int pad[3],
                                   void* stream) {
  if (!plan || plan->elem_bytes != 2) return CONV3D_EINVAL;
  return run_host_impl(plan, x_host, w_host, nullptr, y_host, stride, pad, stream);
}

conv3d_status conv3d_fp8_plan_ex(conv3d_fp8_plan_t* out, int N, int C, int D, int H, int W, int K,
                                 int T, int R, int S, const int stride[3], const int pad[3],
                                 int device, const conv3d_fp8_options* opts) {
  return plan_impl(1, out, N, C, D, H, W, K, T, R, S, stride, pad, device, opts);
}

conv3d_status conv3d_fp8_plan(conv3d_fp8_plan_t* out, int N, int C, int D, int H, int W, int K,
                              int T, int R, int S, const int stride[3], const int pad[3],
                              int device) {
  return plan_impl(1, out, N, C, D, H, W, K, T, R, S, stride, pad, device, nullptr);
}

conv3d_status conv3d_fp8_run(conv3d_fp8_plan_t plan, const void* x, const void* w,
                             const float* scale_x, const float* scale_w, void* y,
                             const int stride[3], const int pad[3], void* stream) {
  if (plan && plan->elem_bytes != 1) return CONV3D_EINVAL;
  return run_impl(plan, x, w, scale_x, scale_w, y, stride, pad, stream);
}

conv3d_status conv3d_bf16_plan_ex(conv3d_fp8_plan_t* out, int N, int C, int D, int H, int W, int K,
                                  int T, int R, int S, const int stride[3], const int pad[3],
                                  int device, const conv3d_fp8_options* opts) {
  return plan_impl(2, out, N, C, D, H, W, K, T, R, S, stride, pad, device, opts);
}

conv3d_status conv3d_bf16_plan(conv3d_fp8_plan_t* out, int N, int C, int D, int H, int W, int K,
                               int T, int R, int S, const int stride[3], const int pad[3],
                               int device) {
  return plan_impl(2, out, N, C, D, H, W, K, T, R, S, stride, pad, device, nullptr);
}

conv3d_status conv3d_bf16_run(conv3d_fp8_plan_t plan, const void* x, const void* w, void* y,
                              const int stride[3], const int pad[3], void* stream) {
  if (!plan || plan->elem_bytes != 2) return CONV3D_EINVAL;
  return run_impl(plan, x, w, plan->ones, plan->ones + 1, y, stride, pad, stream);
}

conv3d_status conv3d_fp8_quantize(const void* src, int src_type, long long n, void* dst_e4m3,
                                  float* scale_out, void* stream) {
  if (!src || !dst_e4m3 || !scale_out || n <= 0) return CONV3D_EINVAL;
  if (src_type != CONV3D_SRC_F32 && src_type != CONV3D_SRC_BF16) return CONV3D_EINVAL;
  if (!aligned(src, 16) || !aligned(dst_e4m3, 16) || !aligned(scale_out, 4)) return CONV3D_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int type = src_type == CONV3D_SRC_F32 ? kSrcF32 : kSrcBf16;
  // scale_out holds the amax bits until the finalisation turns them into the scale
  unsigned* amax = reinterpret_cast<unsigned*>(scale_out);
  if (launch_amax(src, type, n, amax, s) != cudaSuccess ||
      launch_quant_cast(src, type, n, static_cast<uint8_t*>(dst_e4m3), amax, s) != cudaSuccess ||
      launch_quant_finalize(amax, scale_out, nullptr, s) != cudaSuccess)
    return CONV3D_ECUDA;
  return CONV3D_OK;
}

conv3d_status conv3d_fp8_run_quantize_x(conv3d_fp8_plan_t plan, const void* x_src, int src_type,
                                        const void* w, const float* scale_w, void* y,
                                        const int stride[3], const int pad[3], float* scale_x_out,
                                        void* stream) {
  if (!plan || plan->elem_bytes != 1 || plan->p.x_cl) return CONV3D_EINVAL;
  if (src_type != CONV3D_SRC_F32 && src_type != CONV3D_SRC_BF16) return CONV3D_EINVAL;
  if (!x_src || !aligned(x_src, 16) || (scale_x_out && !aligned(scale_x_out, 4)))
    return CONV3D_EINVAL;
  if (!w || !scale_w || !y || !stride || !pad) return CONV3D_EINVAL;
  for (int i = 0; i < 3; ++i)
    if (stride[i] != plan->stride[i] || pad[i] != plan->pad[i]) return CONV3D_EINVAL;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return CONV3D_ECUDA;
  if (cur != plan->device) return CONV3D_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int type = src_type == CONV3D_SRC_F32 ? kSrcF32 : kSrcBf16;
  const ConvParams& q = plan->p;
  const long long n = (long long)q.N * q.C * q.D * q.H * q.W;
  // the plan's 256-byte status slot: status word at 0, amax bits at 64, the scale of x at 68
  uint8_t* slot = reinterpret_cast<uint8_t*>(q.status);
  unsigned* amax = reinterpret_cast<unsigned*>(slot + 64);
  float* scale_x = reinterpret_cast<float*>(slot + 68);
  if (launch_amax(x_src, type, n, amax, s) != cudaSuccess ||
      launch_quant_finalize(amax, scale_x, scale_x_out, s) != cudaSuccess)
    return CONV3D_ECUDA;
  return run_impl(plan, x_src, w, scale_x, scale_w, y, stride, pad, stream, type);
}

conv3d_status conv3d_bf16_describe(int N, int C, int D, int H, int W, int K, int T, int R, int S,
                                   const int stride[3], const int pad[3], int sm_count,
                                   const conv3d_fp8_options* opts, conv3d_fp8_plan_info* info) {
  return decide(2, N, C, D, H, W, K, T, R, S, stride, pad, sm_count, opts, info, nullptr, nullptr);
}

conv3d_status conv3d_fp8_set_timing_events(conv3d_fp8_plan_t plan, void* ev_begin, void* ev_end) {
  if (!plan) return CONV3D_EINVAL;
  plan->ev_begin = static_cast<cudaEvent_t>(ev_begin);
  plan->ev_end = static_cast<cudaEvent_t>(ev_end);
  return CONV3D_OK;
}

conv3d_status conv3d_fp8_set_pack_timing_event(conv3d_fp8_plan_t plan, void* ev_pack) {
  if (!plan) return CONV3D_EINVAL;
  plan->ev_pack = static_cast<cudaEvent_t>(ev_pack);
  return CONV3D_OK;
}

conv3d_status conv3d_fp8_set_write_counter(conv3d_fp8_plan_t plan, void* counts) {
  if (!plan) return CONV3D_EINVAL;
#ifdef C3D_COUNT_WRITES
  if (counts && reinterpret_cast<uintptr_t>(counts) % 4 != 0) return CONV3D_EINVAL;
  plan->p.write_count = static_cast<uint32_t*>(counts);
  return CONV3D_OK;
#else
  (void)counts;
  return CONV3D_EUNSUPPORTED;
#endif
}

conv3d_status conv3d_fp8_check(conv3d_fp8_plan_t plan) {
  if (!plan) return CONV3D_EINVAL;
  DeviceGuard guard;
  if (guard.set(plan->device) != cudaSuccess) return CONV3D_ECUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return CONV3D_ECUDA;
  int status = 0;
  if (cudaMemcpy(&status, plan->p.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CONV3D_ECUDA;
  if (status != 0) {
    cudaMemset(plan->p.status, 0, sizeof(int));
    cudaDeviceSynchronize();
    return CONV3D_EDEVICE;
  }
  return CONV3D_OK;
}

conv3d_status conv3d_fp8_get_info(conv3d_fp8_plan_t plan, conv3d_fp8_plan_info* info) {
  if (!plan || !info) return CONV3D_EINVAL;
  *info = plan->info;
  return CONV3D_OK;
}

size_t conv3d_fp8_workspace_size(conv3d_fp8_plan_t plan) {
  return plan ? plan->info.workspace_bytes : 0;
}

conv3d_status conv3d_fp8_out_dims(conv3d_fp8_plan_t plan, int* Do, int* Ho, int* Wo) {
  if (!plan || !Do || !Ho || !Wo) return CONV3D_EINVAL;
  *Do = plan->info.Do;
  *Ho = plan->info.Ho;
  *Wo = plan->info.Wo;
  return CONV3D_OK;
}

void conv3d_fp8_destroy(conv3d_fp8_plan_t plan) {
  if (!plan) return;
  {
    DeviceGuard guard;
    if (guard.set(plan->device) == cudaSuccess) {
      cudaDeviceSynchronize();
      cudaFree(plan->workspace);
      cudaFree(plan->host_stage);
    }
  }
  delete plan;
}

const char* conv3d_fp8_strerror(conv3d_status s) {
  switch (s) {
    case CONV3D_OK: return "success";
    case CONV3D_EINVAL: return "invalid argument";
    case CONV3D_EUNSUPPORTED: return "unsupported problem or device";
    case CONV3D_ENOMEM: return "device workspace allocation failed";
    case CONV3D_ECUDA: return "CUDA call failed";
    case CONV3D_EDEVICE: return "kernel stopped early: a bounded wait ran out of time";
  }
  return "unknown status";
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot call cudaMalloc: a host framework whose caching allocator owns the device's
// memory pool and forbids stray allocations, a plugin interface that hands a kernel its tensors
// but gives it no way to request memory, or a latency-critical loop that cannot afford the device
// synchronisation that cudaFree implies. conv3d_fp8_run_noalloc serves them: it runs the same
// kernels as conv3d_fp8_run, but its scratch (the packed operands, split-K partials and the status
// word) lives in the fixed-size device array below instead of a plan-owned workspace.
//
// The array is reserved by the CUDA runtime when this library's device code is loaded on a GPU and
// stays reserved until the process exits. Every call on a device shares it and it keeps the last
// call's contents: each call rewrites everything it reads (the pack kernel writes every byte of
// the padded operands, partials are written before they are reduced) and clears the status word
// itself. Two calls whose work overlaps on the GPU (other streams, other host threads) race on the
// array; serialise them.
// ------------------------------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[CONV3D_FP8_NOALLOC_SCRATCH_BYTES];

#include <mutex>

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_base[kNoAllocMaxDevices] = {};
int* g_noalloc_status[kNoAllocMaxDevices] = {};  // status word of the latest call on each device

// Once per device, with that device current: take the device address of the scratch array (the
// host-side symbol is only a stand-in and must never reach a kernel) and grant the main kernel the
// device's opt-in shared memory. Allocates nothing.
conv3d_status noalloc_setup(int dev, void** base) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_base[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return CONV3D_ECUDA;
    }
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        conv_set_smem_attr((size_t)optin) != cudaSuccess) {
      cudaGetLastError();
      return CONV3D_ECUDA;
    }
    g_noalloc_base[dev] = ptr;
  }
  *base = g_noalloc_base[dev];
  return CONV3D_OK;
}

}  // namespace

extern "C" conv3d_status conv3d_fp8_run_noalloc(int N, int C, int D, int H, int W, int K, int T,
                                                int R, int S, const int stride[3],
                                                const int pad[3], const void* x, const void* w,
                                                const float* scale_x, const float* scale_w,
                                                void* y, void* stream) {
  if (!x || !w || !scale_x || !scale_w || !y || !stride || !pad) return CONV3D_EINVAL;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(scale_x, 4) ||
      !aligned(scale_w, 4))
    return CONV3D_EINVAL;
  // Shape errors first, without touching the device.
  conv3d_fp8_plan_info info{};
  conv3d_status st =
      decide(1, N, C, D, H, W, K, T, R, S, stride, pad, 1, nullptr, &info, nullptr, nullptr);
  if (st != CONV3D_OK) return st;

  int dev = -1, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return CONV3D_ECUDA;
  }
  if (dev < 0 || dev >= kNoAllocMaxDevices) return CONV3D_EUNSUPPORTED;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return CONV3D_ECUDA;
  if (major != 10 || minor != 3) return CONV3D_EUNSUPPORTED;

  // the scratch address and the kernels' shared-memory grant, before any occupancy query
  void* base = nullptr;
  st = noalloc_setup(dev, &base);
  if (st != CONV3D_OK) return st;
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return CONV3D_ECUDA;

  ConvParams p{};
  Layout L{};
  st = decide(1, N, C, D, H, W, K, T, R, S, stride, pad, sms, nullptr, &info, &p, &L);
  if (st != CONV3D_OK) return st;
  if (p.pair) {  // plan for the CTA pairs the device can actually hold at once
    const int clusters = conv_pair_max_active_clusters(p);
    if (clusters > 0 && clusters < sms / 2) {
      st = decide(1, N, C, D, H, W, K, T, R, S, stride, pad, sms, nullptr, &info, &p, &L,
                  clusters);
      if (st != CONV3D_OK) return st;
    }
  }
  if (L.total > (size_t)CONV3D_FP8_NOALLOC_SCRATCH_BYTES) return CONV3D_EUNSUPPORTED;
  const size_t smem = p.pair ? conv_pair_smem_bytes(p)
                             : conv_smem_bytes(p.block_n, p.stages, p.epi_tma != 0);
  if ((long long)smem > (long long)optin) return CONV3D_EUNSUPPORTED;

  uint8_t* ws = static_cast<uint8_t*>(base);
  p.xp = L.xp_bytes ? ws + L.xp_off : nullptr;
  p.wp = ws + L.wp_off;
  p.partials = L.part_bytes ? reinterpret_cast<float*>(ws + L.part_off) : nullptr;
  p.status = reinterpret_cast<int*>(ws + L.status_off);
  // the shared scratch holds other problems between calls: the pack writes the halo every run
  p.halo_once = 0;
  p.x = static_cast<const uint8_t*>(x);
  p.w = static_cast<const uint8_t*>(w);
  p.y = static_cast<uint16_t*>(y);
  p.scale_x = scale_x;
  p.scale_w = scale_w;

  if (p.pair) {  // never more clusters than can be resident at once
    const int clusters = conv_pair_max_active_clusters(p);
    if (clusters > 0 && info.grid > 2 * clusters) info.grid = 2 * clusters;
  }
  CUtensorMap wmap{}, xmap{};
  st = encode_maps(&wmap, &xmap, p);
  if (st == CONV3D_OK && p.route == kRouteDirect) st = encode_wmap(&wmap, p, w);
  if (st != CONV3D_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(p.status, 0, sizeof(int), s) != cudaSuccess) return CONV3D_ECUDA;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    g_noalloc_status[dev] = p.status;
  }
  if (launch_pack(p, s) != cudaSuccess) return CONV3D_ECUDA;
  const CUtensorMap ymap{};  // explicit guarded stores here (no TMA-store epilogue)
  if (launch_conv(p, wmap, xmap, ymap, info.row_chk != 0, info.grid, s) != cudaSuccess)
    return CONV3D_ECUDA;
  if (has_split_tiles(p) && launch_splitk_reduce(p, info.row_chk != 0, s) != cudaSuccess)
    return CONV3D_ECUDA;
  return CONV3D_OK;
}

extern "C" conv3d_status conv3d_fp8_noalloc_check(void) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return CONV3D_ECUDA;
  }
  if (dev < 0 || dev >= kNoAllocMaxDevices) return CONV3D_EUNSUPPORTED;
  int* status = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    status = g_noalloc_status[dev];
  }
  if (!status) return CONV3D_OK;  // no allocation-free call on this device yet
  if (cudaDeviceSynchronize() != cudaSuccess) return CONV3D_ECUDA;
  int word = 0;
  if (cudaMemcpy(&word, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CONV3D_ECUDA;
  if (word == 0) return CONV3D_OK;
  if (cudaMemset(status, 0, sizeof(int)) != cudaSuccess) return CONV3D_ECUDA;
  return CONV3D_EDEVICE;
}
