// conv_tc.cu -- the implicit-GEMM main kernel on one CTA: tcgen05 FP8 MMAs (M = 128) with TMEM
// accumulators.
//
// GEMM view (the subject page, "Root cause"): row = output position (npq = N*Do*Ho*Wo rows),
// col = output channel (K columns), reduction over K_gemm = (tap, channel) of T*R*S*C.
//
// One persistent CTA per SM walks a static list of work units (m-tile, n-tile, K-split).
// Warp roles:
//   warps 0-3  epilogue: TMEM -> registers, scale, bf16, stores masked on row < npq and col < K
//              (warp w owns TMEM lanes 32w..32w+31, i.e. rows 32w..32w+31 of the tile)
//   warp 8     TMA loader: per stage one 2D tile of the weights (B: the packed copy, or the
//              caller's KCTRS w on the direct route) and, on the im2col route, the A tile as
//              128/a_cb im2col loads (one per tap and channel block) of 128 consecutive output
//              positions from the channels-last input (the TMA unit zero-fills taps outside the
//              volume and rows past the last image), or on the direct route one 2D tile of the
//              explicit im2col of x (rows past npq and K bytes past K_gemm read zero). Also owns
//              the TMEM allocation.
//   warps 4-7  gather route (C % 32 != 0 or paddings beyond the im2col corner range): A by
//              16-byte cp.async gathers from the zero-padded channels-last input into the
//              128-byte-swizzled stage; rows at or past npq are zero-filled. On the im2col and
//              direct routes A arrives by TMA with B and these warps stay idle (on the direct
//              route A and B are the explicit im2col of x and the caller's KCTRS weights, in the
//              same K order).
//   warp 9     MMA issuer: 4 x tcgen05.mma (M=128, N=block_n, K=32 bytes) per 128-byte K block;
//              kind::f8f6f4 on e4m3 bytes, or kind::f16 on bfloat16 pairs (kBf16): the tiles,
//              stages and descriptors are the same in bytes
// Warps 8 and 9 run their loops on all 32 lanes (every lane waits on the barriers) and issue the
// copies, MMAs and commits of a stage from one lane chosen by elect.sync.
// Stages are handed over with mbarriers: TMA-full (transaction bytes of A and/or B), A-full (128
// gather arrivals, gather route), stage-empty (tcgen05.commit). Two TMEM accumulators let the
// epilogue of one tile overlap the main loop of the next. Every wait is bounded; a wait that runs
// out records a status bit and the whole CTA winds down without faulting.
#include <cuda_runtime.h>

#include "conv_common.cuh"

namespace c3d {

constexpr int kLoaderLag = 2;  // cp.async groups kept in flight before a stage is signalled full

template <bool kRowChk, bool kBf16>
__global__ void __launch_bounds__(kNumThreads, 1)
    conv3d_fp8_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                         const __grid_constant__ CUtensorMap xmap,
                         const __grid_constant__ CUtensorMap ymap, const ConvParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);  // 1024-aligned stages

  const int S = p.stages;
  const uint32_t b_bytes = (uint32_t)p.block_n * kBlockK;
  uint8_t* sA = smem;
  uint8_t* sB = smem + (size_t)S * kATileBytes;
  // bf16 staging of the TMA-store epilogue (1024-aligned, after the stages), then the barriers
  uint16_t* sEpi = reinterpret_cast<uint16_t*>(sB + (size_t)S * b_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + (size_t)S * b_bytes +
                                               (p.epi_tma ? (size_t)kEpiStageBytes : 0));
  // bars: fullA[S], fullB[S], empty[S], accFull[2], accEmpty[2], drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t sA_u32 = smem_u32(sA), sB_u32 = smem_u32(sB);
  const uint32_t bars_u32 = smem_u32(bars);
  auto fullA = [&](int s) { return bars_u32 + 8u * s; };
  auto fullB = [&](int s) { return bars_u32 + 8u * (S + s); };
  auto empty = [&](int s) { return bars_u32 + 8u * (2 * S + s); };
  auto accFull = [&](int b) { return bars_u32 + 8u * (3 * S + b); };
  auto accEmpty = [&](int b) { return bars_u32 + 8u * (3 * S + 2 + b); };
  const uint32_t drain_bar = bars_u32 + 8u * (3 * S + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(fullA(s), 128);
      mbar_init(fullB(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accFull(b), 1);
      mbar_init(accEmpty(b), 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
    tmem_relinquish();
    if (lane == 0) {
      prefetch_tensormap(&wmap);
      if (p.route == kRouteIm2col || p.route == kRouteDirect) prefetch_tensormap(&xmap);
      if (p.epi_tma) prefetch_tensormap(&ymap);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait_primary();        // the pack's output (launched dependent on it), complete and visible
  pdl_launch_dependents();   // the reduction of split tiles may be scheduled
  const AbortState ab{abort_flag, p.status, p.timeout_ns};
  const bool im2col = p.route == kRouteIm2col;
  const bool direct = p.route == kRouteDirect;
  const bool a_tma = im2col || direct;  // A arrives by TMA on the B barrier (no loader warps)

  if (warp < 4) {
    // ------------------------------------------------------------------------------ epilogue
    const float scale = __ldg(p.scale_x) * __ldg(p.scale_w);
    uint32_t tc = 0, chunk = 0;
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++tc) {
      const Unit un = decode_unit(p, u);
      const int buf = tc & 1;
      bool ok = wait_bounded(accFull(buf), (tc >> 1) & 1, ab, kStatusWaitAccFull);
      // the TMA-store epilogue synchronises its 128 threads: they go on or stop together
      if (p.epi_tma) ok = named_barrier_and(1, 128, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t trow =
          tmem_base + (uint32_t)buf * p.acc_stride + ((uint32_t)(warp * 32) << 16);
      if (p.epi_tma && un.part < 0)
        epilogue_tile_tma(p, un, &ymap, trow, un.m_tile * p.block_m, threadIdx.x, scale, sEpi,
                          chunk);
      else
        epilogue_row<kRowChk>(p, un, trow, threadIdx.x, scale, 0, p.block_n);
      tc_fence_before();
      mbar_arrive(accEmpty(buf));
    }
    if (p.epi_tma && threadIdx.x == 0) bulk_wait_group_all();  // stores done before exit
  } else if (warp < 8) {
    // ------------------------------------------------------------------------------ A gather
    if (!a_tma) {
      const int pt = threadIdx.x - 128;
      const int q = pt & 7;    // 16-byte chunk of the 128-byte K block
      const int rb = pt >> 3;  // rows rb, rb+16, ..., rb+112
      const uint32_t row_dst = sA_u32 + (uint32_t)rb * 128u + (uint32_t)((q ^ (rb & 7)) << 4);
      const int RS = p.R * p.S;
      Ring ring;
      uint32_t signaled = 0;
      int inflight = 0;
      bool aborted = false;
      for (int u = blockIdx.x; u < p.num_units && !aborted; u += gridDim.x) {
        const Unit un = decode_unit(p, u);
        long long rowoff[8];
        bool rowok[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int m = un.m_tile * kBlockM + rb + 16 * i;
          rowok[i] = !kRowChk || m < p.npq;
          const int mm = rowok[i] ? m : 0;
          const int n = mm / p.dhw;
          const int pix = mm - n * p.dhw;
          const int wo = pix % p.Wo;
          const int t2 = pix / p.Wo;
          const int ho = t2 % p.Ho;
          const int od = t2 / p.Ho;
          rowoff[i] =
              ((((long long)n * p.Dp + od * p.sd) * p.Hp + ho * p.sh) * p.Wp + wo * p.sw) * p.C;
        }
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          const int stage = ring.stage;
          if (!wait_bounded(empty(stage), ring.phase ^ 1u, ab, kStatusWaitEmpty)) {
            aborted = true;
            break;
          }
          const int kk = kb * kBlockK + q * 16;
          const bool kok = kk < p.kg;
          long long tapoff = 0;
          if (kok) {
            const int tap = kk / p.C;
            const int c = kk - tap * p.C;
            const int t = tap / RS;
            const int rs = tap - t * RS;
            const int r = rs / p.S;
            const int s = rs - r * p.S;
            tapoff = (((long long)t * p.Hp + r) * p.Wp + s) * p.C + c;
          }
          const uint32_t dst = row_dst + (uint32_t)stage * kATileBytes;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const bool ok = kok && rowok[i];
            const uint8_t* src = ok ? p.xp + rowoff[i] + tapoff : p.xp;
            cp_async_16_zfill(dst + (uint32_t)i * 2048u, src, ok ? 16u : 0u);
          }
          cp_async_commit();
          ring.next(S);
          if (++inflight > kLoaderLag) {
            cp_async_wait_group<kLoaderLag>();
            fence_proxy_async_smem();
            mbar_arrive(fullA(signaled % S));
            ++signaled;
            --inflight;
          }
        }
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
      if (!aborted) {
        for (; inflight > 0; --inflight, ++signaled) mbar_arrive(fullA(signaled % S));
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------------------------ TMA loader
    // The whole warp runs the loop and waits on the barriers; one elected lane issues the copies.
    {
      uint32_t it = 0;
      Ring ring;
      const bool skip_first = (p.debug_flags & 1) != 0;
      for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
        const Unit un = decode_unit(p, u);
        StartPixel px{};
        TapWalk walk;
        if (im2col) {
          px.set(p, un.m_tile * kBlockM);  // the TMA walks the next 127 output positions
          walk.start(p, un.kb0 * kBlockK);
        }
        bool aborted = false;
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          const int stage = ring.stage;
          if (!wait_bounded_warp(empty(stage), ring.phase ^ 1u, ab, kStatusWaitEmpty)) {
            aborted = true;
            break;
          }
          const int kk0 = kb * kBlockK;
          const int nsub = im2col ? min(kBlockK, p.kg - kk0) / p.a_cb : 0;
          const bool issue = !(skip_first && it == 0) && elect_one();
          if (issue) {
            mbar_arrive_expect_tx(fullB(stage), b_bytes + (uint32_t)(nsub * p.a_cb * kBlockM) +
                                                    (direct ? (uint32_t)kATileBytes : 0u));
            tma_load_2d(sB_u32 + (uint32_t)stage * b_bytes, &wmap, fullB(stage), kk0,
                        un.n_tile * p.block_n);
            if (direct)  // the full 16 KB box lands (out-of-range rows and bytes as zeros)
              tma_load_2d(sA_u32 + (uint32_t)stage * kATileBytes, &xmap, fullB(stage), kk0,
                          un.m_tile * kBlockM);
          }
          const uint32_t a_dst = sA_u32 + (uint32_t)stage * kATileBytes;
          for (int q = 0; q < nsub; ++q) {
            if (issue)
              tma_load_im2col_5d(a_dst + (uint32_t)(q * kBlockM * p.a_cb), &xmap, fullB(stage),
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
      // Before the CTA may exit, every tile this warp requested must have landed.
      const uint32_t first = it > (uint32_t)S ? it - (uint32_t)S : 0u;
      for (uint32_t j = first; j < it; ++j) {
        if (skip_first && j == 0) continue;
        wait_drain(fullB(j % S), (j / S) & 1, p.timeout_ns, p.status, kStatusWaitDrain);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and waits on the barriers; one elected lane issues the MMAs of
    // a stage together with the commits that track them.
    {
      const uint32_t idesc = make_idesc<kBf16>(kBlockM, (uint32_t)p.block_n);
      // A rows are 128 bytes (SW128) on the gather route, a_cb bytes on the im2col route. K step
      // j covers bytes [32j, 32j+32) of the 128-byte K block: in A it lies in sub-tile 32j / a_cb
      // at byte 32j % a_cb of each row, in B at byte 32j of each 128-byte row. Everything that
      // does not depend on the stage is computed once, so issuing a block is a few adds.
      const uint32_t a_cb = im2col ? (uint32_t)p.a_cb : (uint32_t)kBlockK;
      const uint32_t a_layout =
          a_cb == 128 ? kLayoutSw128 : (a_cb == 64 ? kLayoutSw64 : kLayoutSw32);
      const uint64_t adesc0 = make_kmajor_desc(sA_u32, a_cb, a_layout);
      const uint64_t bdesc0 = make_sw128_kmajor_desc(sB_u32);
      uint32_t a_step[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        a_step[j] =
            (((uint32_t)(j * kMmaK) / a_cb) * kBlockM * a_cb + (uint32_t)(j * kMmaK) % a_cb) >> 4;
      const uint32_t a_stage16 = kATileBytes >> 4, b_stage16 = b_bytes >> 4;
      uint32_t tc = 0;
      Ring ring;
      bool aborted = false;
      for (int u = blockIdx.x; u < p.num_units && !aborted; u += gridDim.x, ++tc) {
        const Unit un = decode_unit(p, u);
        const int buf = tc & 1;
        if (!wait_bounded_warp(accEmpty(buf), ((tc >> 1) & 1) ^ 1, ab, kStatusWaitAccEmpty))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)buf * p.acc_stride;
        for (int kb = un.kb0; kb < un.kb1; ++kb) {
          const int stage = ring.stage;
          const uint32_t ph = ring.phase;
          if ((!a_tma && !wait_bounded_warp(fullA(stage), ph, ab, kStatusWaitFull)) ||
              !wait_bounded_warp(fullB(stage), ph, ab, kStatusWaitFull)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint64_t adesc = adesc0 + (uint64_t)((uint32_t)stage * a_stage16);
            const uint64_t bdesc = bdesc0 + (uint64_t)((uint32_t)stage * b_stage16);
            const uint32_t acc0 = kb > un.kb0 ? 1u : 0u;
            const int rem = p.kg - kb * kBlockK;
            if (rem >= kBlockK) {
              mma_cta<kBf16>(d_tmem, adesc + a_step[0], bdesc, idesc, acc0);
              mma_cta<kBf16>(d_tmem, adesc + a_step[1], bdesc + 2u, idesc, 1u);
              mma_cta<kBf16>(d_tmem, adesc + a_step[2], bdesc + 4u, idesc, 1u);
              mma_cta<kBf16>(d_tmem, adesc + a_step[3], bdesc + 6u, idesc, 1u);
            } else {
              const int nsteps = (rem + kMmaK - 1) / kMmaK;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (j < nsteps)
                  mma_cta<kBf16>(d_tmem, adesc + a_step[j], bdesc + 2u * j, idesc,
                                 j > 0 ? 1u : acc0);
            }
            mma_commit(empty(stage));
            if (kb + 1 == un.kb1) mma_commit(accFull(buf));  // the unit's last stage
          }
          __syncwarp();
          ring.next(S);
        }
        if (aborted) break;
      }
      // Every MMA must be complete before TMEM is released (elect.sync picks the same lane of a
      // converged warp each time, the lane that issued them).
      if (elect_one()) mma_commit(drain_bar);
      __syncwarp();
      wait_drain(drain_bar, 0, p.timeout_ns, p.status, kStatusWaitDrain);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
}

size_t conv_smem_bytes(int block_n, int stages, bool epi_tma) {
  return 1024 + (size_t)stages * (kATileBytes + (size_t)block_n * kBlockK) +
         (epi_tma ? (size_t)kEpiStageBytes : 0) +
         (size_t)(3 * stages + 5) * 8 + 16;
}

cudaError_t conv_set_smem_attr(size_t smem_bytes) {
  const int v = (int)smem_bytes;
  cudaError_t e = cudaSuccess;
  const void* kernels[] = {(const void*)conv3d_fp8_tc_kernel<true, false>,
                           (const void*)conv3d_fp8_tc_kernel<false, false>,
                           (const void*)conv3d_fp8_tc_kernel<true, true>,
                           (const void*)conv3d_fp8_tc_kernel<false, true>};
  for (const void* k : kernels)
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, v);
  if (e == cudaSuccess) e = conv_pair_set_smem_attr(smem_bytes);
  return e;
}

cudaError_t launch_conv(const ConvParams& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                        const CUtensorMap& ymap, bool row_chk, int grid, cudaStream_t stream) {
  if (p.pair) return launch_conv_pair(p, wmap, xmap, ymap, row_chk, grid, stream);
  const size_t smem = conv_smem_bytes(p.block_n, p.stages, p.epi_tma != 0);
  const bool bf16 = p.elem_bytes == 2;
  auto kernel = row_chk ? (bf16 ? conv3d_fp8_tc_kernel<true, true>
                               : conv3d_fp8_tc_kernel<true, false>)
                        : (bf16 ? conv3d_fp8_tc_kernel<false, true>
                               : conv3d_fp8_tc_kernel<false, false>);
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

}  // namespace c3d
