// conv_tc_pair.cu -- the implicit-GEMM main kernel on CTA pairs: tcgen05.mma.cta_group::2 with
// M = 256 rows per unit, 128 per CTA.
//
// Same GEMM view and work units as the one-CTA kernel, with block_m = 256. A cluster of two CTAs
// (on two SMs) owns one unit at a time:
//   - each CTA's TMA warp loads its own 128 A rows and its half of the unit's B tile
//     (block_n / 2 weight rows) into its own shared memory, and completes the LEADER's (rank 0)
//     stage barrier, which the leader's TMA warp armed with both CTAs' transaction bytes;
//   - the leader's MMA warp issues tcgen05.mma.cta_group::2 (M=256, N=block_n, K=32): A rows and B
//     halves are read from both CTAs' shared memory at the same offsets and each CTA's TMEM
//     receives its own 128 accumulator rows; tcgen05.commit multicasts the stage-empty and
//     accumulator-full signals to both CTAs;
//   - each CTA's four epilogue warps drain their own TMEM rows (stores masked on real output rows
//     and col < K) and release the accumulator on the leader's barrier (2 x 128 arrivals). An
//     eight-warp epilogue, warps 4-7 taking half of each row's columns, measured 1% slower on the
//     large layer when every tile used it: those epilogues already overlap the next tile's MMAs.
//     Only the pair's last unit, whose epilogue nothing hides, is split with warps 4-7 (the large
//     layer's step 261.8-262.8 against 263.8-264.9 us, interleaved on one GPU).
// Compared with one CTA per 128-row tile, every SM stores and reads only half of the B tile per
// K block, so shared-memory traffic per MMA cycle drops from 192 to 128 bytes and more stages fit.
//
// kGrid (stride-1 convolutions): the rows of a unit are 256 consecutive positions of the
// zero-padded grid of one image (Dg x Hg x Wg, the input with its pads), so the A rows of tap
// (t, r, s) are the grid positions (t*Hg + r)*Wg + s further on. A stage holds one
// (t, r, channel block): a single TMA load of 128 + S - 1 consecutive grid positions serves the S
// taps along W (their MMA descriptors start s rows into it; the 128-byte swizzle is a function of
// the shared-memory address, so the shifted start reads the rows TMA wrote there), plus the S
// matching B tiles. The load is a 2D tile of a zero-padded channels-last copy when the library
// packs x itself, or an im2col load whose traversal covers the padded grid of the caller's
// unpadded channels-last x (zeros outside the volume) when x comes channels-last. That cuts the
// bytes each SM's TMA unit must bring in per MMA by about a third, which is what bounds the
// output-position route. Rows of the grid that are not outputs (h >= Ho, w >= Wo, d >= Do) are
// computed and never stored.
// kBf16: bfloat16 inputs (tcgen05.mma kind::f16, K = 16 elements) instead of e4m3 (kind::f8f6f4,
// K = 32 elements); every tile, stage and descriptor is the same in bytes.
// Every wait is bounded; a wait that runs out records a status bit and both CTAs wind down.
#include <cuda_runtime.h>

#include "conv_common.cuh"

namespace c3d {

constexpr uint64_t kAbortSettleNs = 2ull * 1000 * 1000;  // let copies in flight land on abort

// Shared-memory footprint of one pipeline stage of the pair kernel (per CTA).
__host__ __device__ inline void pair_stage_bytes(const ConvParams& p, bool grid, uint32_t* a_bytes,
                                                 uint32_t* b_bytes) {
  const uint32_t half_n = (uint32_t)p.block_n / 2;
  if (grid) {
    const uint32_t rows = (uint32_t)kBlockM + (uint32_t)p.S - 1;
    *a_bytes = ((rows * (uint32_t)p.a_cb) + 1023u) & ~1023u;
    *b_bytes = (((uint32_t)p.S * half_n * (uint32_t)p.a_cb) + 1023u) & ~1023u;
  } else {
    *a_bytes = (uint32_t)kATileBytes;
    *b_bytes = half_n * (uint32_t)kBlockK;
  }
}

// Padded-grid route: where the A loads of one CTA's 128 rows of unit `un` start. xrow0 is the
// first grid position as a row of the [N*Dg*Hg*Wg][C] view of the zero-padded copy (2D loads);
// (w0, h0, d0, n0) are the unpadded coordinates the im2col traversal starts from (rows past an
// image's grid continue into the next image, as the traversal does); (tt, tr, cb) is the
// (t, r, channel block) of the unit's first K group.
struct GridStart {
  int xrow0, w0, h0, d0, n0, tt, tr, cb;
};

__device__ __forceinline__ GridStart grid_start(const ConvParams& p, const Unit& un,
                                                int row_base) {
  GridStart s;
  const int n = un.m_tile / p.tiles_per_image;
  const int g0 = (un.m_tile - n * p.tiles_per_image) * p.block_m + row_base;
  s.xrow0 = n * p.Dg * p.Hg * p.Wg + g0;
  const int plane = p.Hg * p.Wg;
  int gd = g0 / plane;
  const int grem = g0 - gd * plane;
  const int gh = grem / p.Wg;
  s.w0 = grem - gh * p.Wg - p.pw;
  s.h0 = gh - p.ph;
  s.n0 = n + gd / p.Dg;
  gd = gd % p.Dg;
  s.d0 = gd - p.pd;
  const int ncb = p.C / p.a_cb;
  const int trg = un.kb0 / ncb;
  s.cb = un.kb0 - trg * ncb;
  s.tt = trg / p.R;
  s.tr = trg - s.tt * p.R;
  return s;
}

template <bool kRowChk, bool kGrid, bool kBf16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kNumThreads, 1)
    conv3d_fp8_tc_pair_kernel(const __grid_constant__ CUtensorMap wmap,
                              const __grid_constant__ CUtensorMap xmap,
                              const __grid_constant__ CUtensorMap ymap, const ConvParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);  // 1024-aligned stages

  const int S = p.stages;
  const int half_n = p.block_n / 2;
  uint32_t a_bytes, b_bytes;  // per stage: A rows, this CTA's half of the B tile(s)
  pair_stage_bytes(p, kGrid, &a_bytes, &b_bytes);
  uint8_t* sA = smem;
  uint8_t* sB = smem + (size_t)S * a_bytes;
  // bf16 staging of the TMA-store epilogue (1024-aligned, after the stages), then the barriers
  uint16_t* sEpi = reinterpret_cast<uint16_t*>(sB + (size_t)S * b_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + (size_t)S * b_bytes +
                                               (p.epi_tma ? (size_t)kEpiStageBytes : 0));
  // bars: full[S] (leader's is used), empty[S], accFull[2], accEmpty[2] (leader's), drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // last-unit hand-off to warps 4-7: the TMEM buffer of the pair's last unit, or -1 (none, or
  // the epilogue stopped early)
  volatile int* last_buf = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const uint32_t sA_u32 = smem_u32(sA), sB_u32 = smem_u32(sB);
  const uint32_t bars_u32 = smem_u32(bars);
  auto full = [&](int s) { return bars_u32 + 8u * s; };
  auto empty = [&](int s) { return bars_u32 + 8u * (S + s); };
  auto accFull = [&](int b) { return bars_u32 + 8u * (2 * S + b); };
  auto accEmpty = [&](int b) { return bars_u32 + 8u * (2 * S + 2 + b); };
  const uint32_t drain_bar = bars_u32 + 8u * (2 * S + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t leader_bars = map_to_cta(bars_u32, 0);  // the leader's barriers, cluster window
  const int cluster_id = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;
  const int row_base = (int)rank * kBlockM;  // this CTA's rows within the 256-row unit

  // The TMA warp's first unit and where its loads start, computed before the set-up barriers:
  // the first reads of the kernel parameters and the integer divisions then overlap the barrier
  // initialisation, the TMEM allocation (done by the MMA warp) and the cluster barrier, instead
  // of delaying the first copy by about a microsecond after them.
  Unit tma_un0{};
  GridStart tma_gs0{};
  if (warp == 8 && cluster_id < p.num_units) {
    tma_un0 = decode_unit(p, cluster_id);
    if (kGrid) tma_gs0 = grid_start(p, tma_un0, row_base);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accFull(b), 1);
      mbar_init(accEmpty(b), 2 * 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *last_buf = -1;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc_pair(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
    tmem_relinquish_pair();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tensormap(&wmap);
    prefetch_tensormap(&xmap);
    if (p.epi_tma) prefetch_tensormap(&ymap);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before anyone signals across the pair
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait_primary();        // the pack's output (launched dependent on it), complete and visible
  pdl_launch_dependents();   // the reduction of split tiles may be scheduled
  const AbortState ab{abort_flag, p.status, p.timeout_ns};

  // The last unit's epilogue is not hidden behind any MMA: unless the TMA-store epilogue is on,
  // warps 4-7 take the second half of its columns. Warps 0-3 hand it over at named barrier 3
  // (256 threads), which they reach exactly once on every path: at the last unit, or on their
  // way out when there is none or they stopped early.
  const bool split_last = !p.epi_tma && p.block_n >= 64;
  if (warp < 4) {
    // ------------------------------------------------------------------------------ epilogue
    const float scale = __ldg(p.scale_x) * __ldg(p.scale_w);
    uint32_t tc = 0, chunk = 0;
    bool handed = false;
    for (int u = cluster_id; u < p.num_units; u += num_clusters, ++tc) {
      const Unit un = decode_unit(p, u);
      const int buf = tc & 1;
      const bool last = u + num_clusters >= p.num_units;
      bool ok = wait_bounded<true>(accFull(buf), (tc >> 1) & 1, ab, kStatusWaitAccFull);
      // the TMA-store epilogue and the hand-off synchronise the 128 threads: they go on or stop
      // together
      if (p.epi_tma || split_last) ok = named_barrier_and(1, 128, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t trow =
          tmem_base + (uint32_t)buf * p.acc_stride + ((uint32_t)(warp * 32) << 16);
      int cc1 = p.block_n;
      if (split_last && last) {
        if (threadIdx.x == 0) *last_buf = buf;
        named_barrier_sync(3, 256);
        handed = true;
        cc1 = (p.block_n / 2 + 31) & ~31;
      }
      if (!kGrid && p.epi_tma && un.part < 0)
        epilogue_tile_tma(p, un, &ymap, trow, un.m_tile * p.block_m + row_base, threadIdx.x,
                          scale, sEpi, chunk);
      else
        epilogue_row<kRowChk>(p, un, trow, row_base + threadIdx.x, scale, 0, cc1);
      tc_fence_before();
      mbar_arrive_cluster(leader_bars + (accEmpty(buf) - bars_u32));
    }
    if (split_last && !handed) named_barrier_arrive(3, 256);  // nothing handed over
    if (p.epi_tma && threadIdx.x == 0) bulk_wait_group_all();  // stores done before exit
  } else if (warp < 8) {
    // ------------------------------------------------------------------- last-unit epilogue
    if (split_last) {
      int last_u = -1;
      for (int u = cluster_id; u < p.num_units; u += num_clusters) last_u = u;
      named_barrier_sync(3, 256);
      const int buf = *last_buf;
      if (last_u >= 0 && buf >= 0) {
        tc_fence_after();
        const Unit un = decode_unit(p, last_u);
        const float scale = __ldg(p.scale_x) * __ldg(p.scale_w);
        const uint32_t trow = tmem_base + (uint32_t)buf * p.acc_stride +
                              ((uint32_t)((warp - 4) * 32) << 16);
        epilogue_row<kRowChk>(p, un, trow, row_base + threadIdx.x - 128, scale,
                              (p.block_n / 2 + 31) & ~31, p.block_n);
        tc_fence_before();
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------------------------ TMA loader
    // The whole warp runs the loop and waits on the barriers; one elected lane issues the copies.
    {
      uint32_t it = 0;
      Ring ring;
      const bool skip_first = (p.debug_flags & 1) != 0;
      for (int u = cluster_id; u < p.num_units; u += num_clusters) {
        const Unit un = u == cluster_id ? tma_un0 : decode_unit(p, u);
        bool aborted = false;
        if (kGrid) {
          const GridStart gs = u == cluster_id ? tma_gs0 : grid_start(p, un, row_base);
          const int xrow0 = gs.xrow0, w0 = gs.w0, h0 = gs.h0, d0 = gs.d0, n0 = gs.n0;
          const int ncb = p.C / p.a_cb;
          int tt = gs.tt, tr = gs.tr, cb = gs.cb;  // (t, r, channel block) of the current group
          const uint32_t tx = 2u * ((uint32_t)(kBlockM + p.S - 1) * (uint32_t)p.a_cb +
                                    (uint32_t)(p.S * half_n * p.a_cb));
          for (int g = un.kb0; g < un.kb1; ++g) {
            const int stage = ring.stage;
            if (!wait_bounded_warp<true>(empty(stage), ring.phase ^ 1u, ab, kStatusWaitEmpty)) {
              aborted = true;
              break;
            }
            if (!(skip_first && it == 0) && elect_one()) {
              const uint32_t bar = leader_bars + (full(stage) - bars_u32);
              if (leader) mbar_arrive_expect_tx(full(stage), tx);
              const int c0 = cb * p.a_cb;
              if (p.a_grid_im2col)
                tma_load_im2col_5d_pair(sA_u32 + (uint32_t)stage * a_bytes, &xmap, bar, c0, w0,
                                        h0, d0, n0, 0, (uint16_t)tr, (uint16_t)tt);
              else
                tma_load_2d_pair(sA_u32 + (uint32_t)stage * a_bytes, &xmap, bar, c0,
                                 xrow0 + (tt * p.Hg + tr) * p.Wg);
              const int k_tap0 = ((tt * p.R + tr) * p.S) * p.C + c0;
              const uint32_t b_dst = sB_u32 + (uint32_t)stage * b_bytes;
              for (int ss = 0; ss < p.S; ++ss)
                tma_load_2d_pair(b_dst + (uint32_t)(ss * half_n * p.a_cb), &wmap, bar,
                                 k_tap0 + ss * p.C, un.n_tile * p.block_n + (int)rank * half_n);
            }
            __syncwarp();
            if (++cb == ncb) {
              cb = 0;
              if (++tr == p.R) {
                tr = 0;
                ++tt;
              }
            }
            ++it;
            ring.next(S);
          }
          if (aborted) break;
          continue;
        }
        StartPixel px{};
        px.set(p, un.m_tile * p.block_m + row_base);  // the TMA walks the next 127 positions
        TapWalk walk;
        walk.start(p, un.kb0 * kBlockK);
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          const int stage = ring.stage;
          if (!wait_bounded_warp<true>(empty(stage), ring.phase ^ 1u, ab, kStatusWaitEmpty)) {
            aborted = true;
            break;
          }
          const int kk0 = kb * kBlockK;
          const int nsub = min(kBlockK, p.kg - kk0) / p.a_cb;
          const bool issue = !(skip_first && it == 0) && elect_one();
          const uint32_t bar = leader_bars + (full(stage) - bars_u32);
          if (issue) {
            if (leader)  // arm the stage with the bytes of both CTAs' copies
              mbar_arrive_expect_tx(full(stage),
                                    2u * (b_bytes + (uint32_t)(nsub * p.a_cb * kBlockM)));
            tma_load_2d_pair(sB_u32 + (uint32_t)stage * b_bytes, &wmap, bar, kk0,
                             un.n_tile * p.block_n + (int)rank * half_n);
          }
          const uint32_t a_dst = sA_u32 + (uint32_t)stage * a_bytes;
          for (int q = 0; q < nsub; ++q) {
            if (issue)
              tma_load_im2col_5d_pair(a_dst + (uint32_t)(q * kBlockM * p.a_cb), &xmap, bar,
                                      walk.c, px.w, px.h, px.d, px.n, (uint16_t)walk.s,
                                      (uint16_t)walk.r, (uint16_t)walk.t);
            walk.next(p);
          }
          __syncwarp();
          ++it;
          ring.next(S);
        }
        if (aborted) break;
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and waits on the barriers; one elected lane issues the MMAs of
    // a stage together with the commits that track them.
    if (leader) {
      const uint32_t idesc = make_idesc<kBf16>(2 * kBlockM, (uint32_t)p.block_n);
      const uint32_t a_cb = (uint32_t)p.a_cb;
      const uint32_t a_layout =
          a_cb == 128 ? kLayoutSw128 : (a_cb == 64 ? kLayoutSw64 : kLayoutSw32);
      const uint64_t adesc0 = make_kmajor_desc(sA_u32, a_cb, a_layout);
      const uint64_t bdesc0 = make_sw128_kmajor_desc(sB_u32);
      const uint64_t bdesc_g0 = make_kmajor_desc(sB_u32, a_cb, a_layout);  // grid route's B
      uint32_t a_step[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        a_step[j] =
            (((uint32_t)(j * kMmaK) / a_cb) * kBlockM * a_cb + (uint32_t)(j * kMmaK) % a_cb) >> 4;
      const uint32_t a_stage16 = a_bytes >> 4, b_stage16 = b_bytes >> 4;
      // padded-grid route: tap s starts s rows (s * a_cb bytes) into the A tile and at
      // s * half_n * a_cb bytes in the B stage; K step j adds 32 j bytes to both
      const uint32_t steps_cb = a_cb / kMmaK;
      const uint32_t b_tap16 = ((uint32_t)half_n * a_cb) >> 4, a_row16 = a_cb >> 4;
      uint32_t tc = 0;
      Ring ring;
      bool aborted = false;
      for (int u = cluster_id; u < p.num_units && !aborted; u += num_clusters, ++tc) {
        const Unit un = decode_unit(p, u);
        const int buf = tc & 1;
        if (!wait_bounded_warp<true>(accEmpty(buf), ((tc >> 1) & 1) ^ 1, ab,
                                     kStatusWaitAccEmpty))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)buf * p.acc_stride;
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          const int stage = ring.stage;
          if (!wait_bounded_warp<true>(full(stage), ring.phase, ab, kStatusWaitFull)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint64_t adesc = adesc0 + (uint64_t)((uint32_t)stage * a_stage16);
            const uint32_t acc0 = kb > un.kb0 ? 1u : 0u;
            if (kGrid) {
              // The issuing thread must keep pace with the tensor pipe (one N=256 MMA per 128
              // cycles): per tap, the K steps go out as straight-line code with constant descriptor
              // offsets, and the per-tap offsets advance by one add each.
              uint64_t a_tap = adesc;
              uint64_t b_tap = bdesc_g0 + (uint64_t)((uint32_t)stage * b_stage16);
              uint32_t acc = acc0;
              for (int ss = 0; ss < p.S; ++ss) {
                if (steps_cb == 4) {
                  mma_pair<kBf16>(d_tmem, a_tap, b_tap, idesc, acc);
                  mma_pair<kBf16>(d_tmem, a_tap + 2u, b_tap + 2u, idesc, 1u);
                  mma_pair<kBf16>(d_tmem, a_tap + 4u, b_tap + 4u, idesc, 1u);
                  mma_pair<kBf16>(d_tmem, a_tap + 6u, b_tap + 6u, idesc, 1u);
                } else if (steps_cb == 2) {
                  mma_pair<kBf16>(d_tmem, a_tap, b_tap, idesc, acc);
                  mma_pair<kBf16>(d_tmem, a_tap + 2u, b_tap + 2u, idesc, 1u);
                } else {
                  mma_pair<kBf16>(d_tmem, a_tap, b_tap, idesc, acc);
                }
                acc = 1u;
                a_tap += a_row16;
                b_tap += b_tap16;
              }
            } else {
              const uint64_t bdesc = bdesc0 + (uint64_t)((uint32_t)stage * b_stage16);
              const int rem = p.kg - kb * kBlockK;
              if (rem >= kBlockK) {
                mma_pair<kBf16>(d_tmem, adesc + a_step[0], bdesc, idesc, acc0);
                mma_pair<kBf16>(d_tmem, adesc + a_step[1], bdesc + 2u, idesc, 1u);
                mma_pair<kBf16>(d_tmem, adesc + a_step[2], bdesc + 4u, idesc, 1u);
                mma_pair<kBf16>(d_tmem, adesc + a_step[3], bdesc + 6u, idesc, 1u);
              } else {
                const int nsteps = (rem + kMmaK - 1) / kMmaK;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  if (j < nsteps)
                    mma_pair<kBf16>(d_tmem, adesc + a_step[j], bdesc + 2u * j, idesc,
                                    j > 0 ? 1u : acc0);
              }
            }
            mma_commit_pair(empty(stage), 0x3);
            if (kb + 1 == un.kb1) mma_commit_pair(accFull(buf), 0x3);  // the unit's last stage
          }
          __syncwarp();
          ring.next(S);
        }
        if (aborted) break;
      }
      // Every MMA of the pair must be complete before TMEM is released (elect.sync picks the
      // same lane of a converged warp each time, the lane that issued them).
      if (elect_one()) mma_commit_pair(drain_bar, 0x1);
      __syncwarp();
      wait_drain(drain_bar, 0, p.timeout_ns, p.status, kStatusWaitDrain);
    }
    __syncwarp();
  }

  if (*abort_flag) sleep_ns_bounded(kAbortSettleNs);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the other may still signal or read its memory
  tc_fence_after();
  if (warp == 9) tmem_dealloc_pair(tmem_base, (uint32_t)p.tmem_cols);
}

size_t conv_pair_smem_bytes(const ConvParams& p) {
  uint32_t a_bytes, b_bytes;
  pair_stage_bytes(p, p.route == kRouteGrid, &a_bytes, &b_bytes);
  return 1024 + (size_t)p.stages * (a_bytes + b_bytes) + (p.epi_tma ? (size_t)kEpiStageBytes : 0) +
         (size_t)(2 * p.stages + 5) * 8 + 16;
}

cudaError_t conv_pair_set_smem_attr(size_t smem_bytes) {
  const int v = (int)smem_bytes;
  cudaError_t e = cudaSuccess;
  const void* kernels[] = {(const void*)conv3d_fp8_tc_pair_kernel<true, false, false>,
                           (const void*)conv3d_fp8_tc_pair_kernel<false, false, false>,
                           (const void*)conv3d_fp8_tc_pair_kernel<true, true, false>,
                           (const void*)conv3d_fp8_tc_pair_kernel<true, false, true>,
                           (const void*)conv3d_fp8_tc_pair_kernel<false, false, true>,
                           (const void*)conv3d_fp8_tc_pair_kernel<true, true, true>};
  for (const void* k : kernels)
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, v);
  return e;
}

template <bool kBf16>
cudaError_t launch_pair_typed(const ConvParams& p, const CUtensorMap& wmap,
                              const CUtensorMap& xmap, const CUtensorMap& ymap, bool row_chk,
                              int grid, size_t smem, cudaStream_t stream) {
  auto kernel = p.route == kRouteGrid  // grid rows that are not outputs always need the row test
                    ? conv3d_fp8_tc_pair_kernel<true, true, kBf16>
                    : (row_chk ? conv3d_fp8_tc_pair_kernel<true, false, kBf16>
                               : conv3d_fp8_tc_pair_kernel<false, false, kBf16>);
  // programmatic dependent launch: the prologue overlaps the tail of the pack kernel before it
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kNumThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, wmap, xmap, ymap, p);
}

cudaError_t launch_conv_pair(const ConvParams& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                             const CUtensorMap& ymap, bool row_chk, int grid,
                             cudaStream_t stream) {
  const size_t smem = conv_pair_smem_bytes(p);
  if (p.elem_bytes == 2)
    return launch_pair_typed<true>(p, wmap, xmap, ymap, row_chk, grid, smem, stream);
  return launch_pair_typed<false>(p, wmap, xmap, ymap, row_chk, grid, smem, stream);
}

int conv_pair_max_active_clusters(const ConvParams& p) {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kNumThreads, 1, 1);
  cfg.dynamicSmemBytes = conv_pair_smem_bytes(p);
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, conv3d_fp8_tc_pair_kernel<true, false, false>, &cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace c3d
