// conv_common.cuh -- device pieces shared by the one-CTA and the CTA-pair implicit-GEMM kernels
// and by the split-K reduction.
#pragma once
#include <cuda_bf16.h>

#include "conv3d_fp8_internal.h"
#include "ptx.cuh"

namespace c3d {

// One work unit: an M tile of block_m rows, an N tile of block_n channels and a slice [kb0, kb1)
// of the K blocks. A launch's unit u is the plan's unit unit_base + u. The first full_tiles units
// are whole tiles (part = -1); after them come the
// remaining tiles, each split `splits` ways along K, split-fastest (part = index of the unit's
// fp32 partial slice). Tiles are numbered n-tile fastest.
struct Unit {
  int tile, m_tile, n_tile, split, kb0, kb1, part;
};

__device__ __forceinline__ Unit decode_unit(const ConvParams& p, int u) {
  Unit r;
  u += p.unit_base;  // the launch's units are a contiguous range of the plan's
  if (u < p.full_tiles) {
    r.tile = u;
    r.split = 0;
    r.part = -1;
    r.kb0 = 0;
    r.kb1 = p.k_blocks;
  } else {
    r.part = u - p.full_tiles;
    r.split = r.part % p.splits;
    r.tile = p.full_tiles + r.part / p.splits;
    r.kb0 = r.split * p.kb_per_split;
    r.kb1 = min(r.kb0 + p.kb_per_split, p.k_blocks);
  }
  r.n_tile = r.tile % p.n_tiles;
  r.m_tile = r.tile / p.n_tiles;
  return r;
}

// Position in the ring of S pipeline stages: stage index and the parity of its current phase.
struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int S) {
    if (++stage == S) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

// Wait used only while winding down: ignores the abort flag, still bounded.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                           int* status, int code) {
  if (mbar_try_wait_cluster(bar, parity)) return;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (!mbar_try_wait_cluster(bar, parity)) {
    if ((++spins & 63u) == 0 && globaltimer_ns() - t0 > timeout_ns) {
      atomicOr(status, code);
      return;
    }
  }
}

// Busy-wait for `ns` nanoseconds (used only on the abort path, to let copies in flight land).
__device__ __forceinline__ void sleep_ns_bounded(uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < ns) {
  }
}

// Where accumulator row `row_in_tile` of M tile `m_tile` lands in y: whether it is a real output
// and the NCDHW offset of its channel-0 element (channel k adds k * dhw).
//  - output-position routes: row m = m_tile * block_m + row_in_tile is output position m of the
//    GEMM view; it is real iff m < npq (the row guard of the subject page);
//  - padded-grid route: rows index the zero-padded grid of one image, tile by tile
//    (tiles_per_image tiles per image, none straddling two images); position (d, h, w) of that grid
//    is real iff d < Do, h < Ho and w < Wo.
struct RowDest {
  bool valid;
  long long y_off;
};
__device__ __forceinline__ RowDest row_dest(const ConvParams& p, int m_tile, int row_in_tile) {
  RowDest r;
  if (p.route == kRouteGrid) {
    const int n = m_tile / p.tiles_per_image;
    const int mg = (m_tile - n * p.tiles_per_image) * p.block_m + row_in_tile;
    const int hw = p.Hg * p.Wg;
    const int d = mg / hw;
    const int rem = mg - d * hw;
    const int h = rem / p.Wg;
    const int w = rem - h * p.Wg;
    r.valid = d < p.Do && h < p.Ho && w < p.Wo;
    r.y_off = r.valid ? (long long)n * p.K * p.dhw + ((long long)d * p.Ho + h) * p.Wo + w : 0;
  } else {
    const int m = m_tile * p.block_m + row_in_tile;
    r.valid = m < p.npq;
    const int n = m / p.dhw;
    r.y_off = r.valid ? (long long)n * p.K * p.dhw + (m - n * p.dhw) : 0;
  }
  return r;
}

// Write counting, in a library built with C3D_COUNT_WRITES (a test build: every store of output
// element i also adds one to write_count[i], so a test can check that each element is written
// exactly once); the product build compiles it to nothing.
__device__ __forceinline__ void count_write(const ConvParams& p, long long i) {
#ifdef C3D_COUNT_WRITES
  if (p.write_count) atomicAdd(p.write_count + i, 1u);
#else
  (void)p;
  (void)i;
#endif
}

// Epilogue of one thread: columns [cc0, cc1) (multiples of 32) of its accumulator row (TMEM lane)
// of one unit, `trow` = TMEM address of the row's first column in the current buffer.
// `row_in_tile` is the row within the unit's block_m rows. A whole tile: y = bf16(acc * scale),
// stored only if the row is a real output and col < K. A split unit: the raw fp32 row goes to the
// unit's slice of the partials, [part][block_n][block_m]. kRowChk = false compiles the row test
// out (every row real).
template <bool kRowChk>
__device__ __forceinline__ void epilogue_row(const ConvParams& p, const Unit& un, uint32_t trow,
                                             int row_in_tile, float scale, int cc0, int cc1) {
  const int n0 = un.n_tile * p.block_n;
  if (un.part < 0) {
    const RowDest dst = row_dest(p, un.m_tile, row_in_tile);
    const bool row_ok = !kRowChk || dst.valid;
    uint16_t* ybase = p.y + dst.y_off;
    for (int cc = cc0; cc < cc1; cc += 32) {
      if (n0 + cc >= p.K) break;  // warp-uniform
      uint32_t r[32];
      tmem_ld_32x32b_x32(trow + cc, r);
      tmem_ld_wait();
      if (row_ok) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int col = n0 + cc + j;
          if (col < p.K) {
            const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(r[j]) * scale);
            ybase[(long long)col * p.dhw] = *reinterpret_cast<const uint16_t*>(&b);
            count_write(p, dst.y_off + (long long)col * p.dhw);
          }
        }
      }
    }
  } else {
    float* dst = p.partials + ((long long)un.part * p.block_n) * p.block_m + row_in_tile;
    for (int cc = cc0; cc < cc1; cc += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(trow + cc, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j)
        __stcg(dst + (long long)(cc + j) * p.block_m, __uint_as_float(r[j]));
    }
  }
}

// Hardware-bounded epilogue of a whole tile (output-position routes, no split): the 128 epilogue
// threads of the CTA stage 32 columns at a time as bf16 [32 columns][128 rows] in shared memory
// and one thread stores the box with TMA through the tensor map of y viewed as [N][K][dhw]. The
// map's extents bound the store in hardware: rows past the end of image n0 (pix >= dhw), among
// them the padded rows of the last tile, and columns >= K are not written, the TMA counterpart of
// the buffer-descriptor bound of the subject page ("Root cause"). Rows that spill into a later
// image take the explicit guarded stores. Two 8 KB buffers alternate; `chunk` counts the boxes
// this CTA has staged (the same in all 128 threads) and picks the buffer. `m0` = GEMM row of the
// CTA's first row, `row` = this thread's row (0..127). Uses named barrier 1.
__device__ __forceinline__ void epilogue_tile_tma(const ConvParams& p, const Unit& un,
                                                  const CUtensorMap* ymap, uint32_t trow, int m0,
                                                  int row, float scale, uint16_t* stage,
                                                  uint32_t& chunk) {
  const bool any = m0 < p.npq;  // a CTA whose rows are all padding stores nothing
  const int n0 = any ? m0 / p.dhw : 0;
  const int pix0 = m0 - n0 * p.dhw;
  const int r1 = p.dhw - pix0;  // rows [0, r1) lie in image n0
  const int m = m0 + row;
  const bool spill = row >= r1 && m < p.npq;
  long long y_off = 0;
  if (spill) {
    const int n = m / p.dhw;
    y_off = (long long)n * p.K * p.dhw + (m - n * p.dhw);
  }
  const int col0 = un.n_tile * p.block_n;
  for (int cc = 0; cc < p.block_n; cc += 32) {
    if (col0 + cc >= p.K) break;  // uniform across the 128 threads
    uint32_t r[32];
    tmem_ld_32x32b_x32(trow + cc, r);
    tmem_ld_wait();
    uint16_t* buf = stage + (chunk & 1u) * (32 * kBlockM);
    if (chunk >= 2) {  // the box stored from this buffer two chunks ago must have been read:
      // every chunk commits one group, so all but the newest having read covers it
      if (threadIdx.x == 0) bulk_wait_group_read<1>();
      named_barrier_sync(1, 128);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(r[j]) * scale);
      const uint16_t v = *reinterpret_cast<const uint16_t*>(&b);
      buf[j * kBlockM + row] = v;
      if (spill && col0 + cc + j < p.K) {
        p.y[y_off + (long long)(col0 + cc + j) * p.dhw] = v;
        count_write(p, y_off + (long long)(col0 + cc + j) * p.dhw);
      }
    }
    fence_proxy_async_smem();  // the staged values, visible to the TMA unit
    named_barrier_sync(1, 128);
    if (threadIdx.x == 0) {
      if (any) tma_store_3d(ymap, smem_u32(buf), pix0, col0 + cc, n0);
      bulk_commit_group();  // a group per chunk, empty for a tile whose rows are all padding
    }
#ifdef C3D_COUNT_WRITES
    // the box's elements the TMA unit writes: rows of image n0 (pix < dhw), columns < K
    if (any && pix0 + row < p.dhw)
      for (int j = 0; j < 32 && col0 + cc + j < p.K; ++j)
        count_write(p, ((long long)n0 * p.K + col0 + cc + j) * p.dhw + pix0 + row);
#endif
    ++chunk;
  }
}

// The (tap, channel) walk of the im2col loads, in K_gemm order: channel fastest by a_cb, then
// s, r, t.
struct TapWalk {
  int c = 0, s = 0, r = 0, t = 0;
  __device__ __forceinline__ void start(const ConvParams& p, int kk) {
    const int tap = kk / p.C;
    c = kk - tap * p.C;
    const int RS = p.R * p.S;
    t = tap / RS;
    const int rs = tap - t * RS;
    r = rs / p.S;
    s = rs - r * p.S;
  }
  __device__ __forceinline__ void next(const ConvParams& p) {
    c += p.a_cb;
    if (c == p.C) {
      c = 0;
      if (++s == p.S) {
        s = 0;
        if (++r == p.R) {
          r = 0;
          ++t;
        }
      }
    }
  }
};

// im2col start pixel (w, h, d, n) of output position m: the filter window's corner.
struct StartPixel {
  int w, h, d, n;
  __device__ __forceinline__ void set(const ConvParams& p, int m) {
    n = m / p.dhw;
    const int pix = m - n * p.dhw;
    const int ow = pix % p.Wo;
    const int t2 = pix / p.Wo;
    w = ow * p.sw - p.pw;
    h = (t2 % p.Ho) * p.sh - p.ph;
    d = (t2 / p.Ho) * p.sd - p.pd;
  }
};

}  // namespace c3d
