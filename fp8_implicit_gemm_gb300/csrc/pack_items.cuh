// pack_items.cuh -- the items of the operand pack (x NCDHW -> channels-last copy, w KCTRS ->
// K x taps x C): PackPlan (the index ranges of the work) and pack_item (one item).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "conv_common.cuh"

namespace c3d {

// Work of the item path of the pack, as consecutive index ranges of one grid-stride loop:
//   [0, x_items)          interior of x, where the tiled transpose (pack.cu) does not take it:
//                         e4m3 bytes with W % 4 == 0 in items of 16 channels x 4 pixels (16
//                         aligned 4-byte loads, a byte transpose in registers, four 16-byte
//                         stores; 16 pixels with 16-byte loads when W % 16 == 0), else 16
//                         channels x 1 pixel; a bfloat16 x (the BF16 twin) in items of 8
//                         channels x 8 pixels (W % 8 == 0; 16-byte loads), else 8 channels x 2
//                         pixels (x 1 when W is odd); a channels-last x copied in
//                         16-byte chunks into the padded copy (no items when the TMA routes read
//                         that x directly). An fp32 / bfloat16 x quantised to e4m3 on the way is
//                         always transposed by the tiled kernel; its item loop starts at x_items.
//   + halo_row_items      16-byte zero chunks of the padded rows (d or h in the halo)
//   + halo_side_items     16-byte zero chunks of the W-halo pixels of interior rows
//   + w_items             16 channels of one tap of one filter
// Pixels (or pixel groups) run fastest across threads, so each load of a warp is a contiguous run
// along W of the NCDHW input; with 16 or more 16-byte channel chunks a pixel, the 16-pixel items
// run their channel chunk fastest instead, so that each store of a warp writes whole pixel rows
// of the channels-last copy.
constexpr long long kWTileBytes = 16384;  // shared-memory buffer of one weight tile

struct PackPlan {
  long long x_items, halo_row_items, halo_side_items, w_items;
  // Weights by tiles (pack_w_tile) when a 16-byte column of every tap fits the tile buffer: one
  // block per (filter k, w_group 16-byte channel chunks); w_items is then 0.
  long long w_blocks;
  int w_group;
  bool hex;   // e4m3 bytes and W % 16 == 0: 16-pixel items (16-byte loads)
  bool quad;  // e4m3 and W % 4 == 0: 4-pixel items
  bool oct;   // bfloat16 and W % 8 == 0: 8-pixel items (16-byte loads)
  bool two;   // bfloat16 and W % 2 == 0: 2-pixel items
  bool copy;  // x is channels-last already: 16-byte chunk copies
  bool cfast; // hex or oct items with the channel chunk fastest across threads (>= 16 chunks a
              // pixel):
              // a warp's stores of one instruction cover whole pixel rows (C = 256: large layer
              // step 262.4 -> 260.9 us); below 16 chunks the pixel-group-fastest order measured
              // faster (vae layer, C = 128: 32.3 against 33.6 us)
};

__host__ __device__ inline PackPlan pack_plan(const ConvParams& p) {
  PackPlan q;
  const long long cq = p.C / 16;
  q.copy = p.x_cl != 0;
  q.quad = !q.copy && p.elem_bytes == 1 && (p.W % 4) == 0;
  q.hex = q.quad && (p.W % 16) == 0;
  q.two = !q.copy && p.elem_bytes == 2 && (p.W % 2) == 0;
  q.oct = q.two && (p.W % 8) == 0;
  q.cfast = (q.hex || q.oct) && cq >= 16;
  const int per_row = q.hex ? p.W / 16 : q.quad ? p.W / 4 : q.oct ? p.W / 8 : (q.two ? p.W / 2 : p.W);
  q.x_items = p.xp == nullptr ? 0 : (long long)p.N * p.D * p.H * cq * per_row;
  const long long halo_rows_per_image = (long long)p.Dp * p.Hp - (long long)p.D * p.H;
  q.halo_row_items = (long long)p.N * halo_rows_per_image * p.Wp * cq;
  q.halo_side_items = (long long)p.N * p.D * p.H * (p.Wp - p.W) * cq;
  q.w_items = (long long)p.K * p.taps * cq;
  q.w_blocks = 0;
  q.w_group = 0;
  if (16LL * p.taps <= kWTileBytes) {
    q.w_group = (int)(kWTileBytes / (16LL * p.taps));
    if (q.w_group > cq) q.w_group = (int)cq;
    q.w_blocks = (long long)p.K * ((cq + q.w_group - 1) / q.w_group);
    q.w_items = 0;
  }
  if (p.halo_once) {  // the plan zeroed its padded copy once: the halo is never written again
    q.halo_row_items = 0;
    q.halo_side_items = 0;
  }
  return q;
}

// Byte transpose of a 4x4 block: v[c] holds pixels 0..3 of channel c; o[j] gets channels 0..3 of
// pixel j.
__device__ __forceinline__ void transpose4x4(const uint32_t v[4], uint32_t o[4]) {
  const uint32_t t0 = __byte_perm(v[0], v[1], 0x5140), t1 = __byte_perm(v[2], v[3], 0x5140);
  const uint32_t t2 = __byte_perm(v[0], v[1], 0x7362), t3 = __byte_perm(v[2], v[3], 0x7362);
  o[0] = __byte_perm(t0, t1, 0x5410);
  o[1] = __byte_perm(t0, t1, 0x7632);
  o[2] = __byte_perm(t2, t3, 0x5410);
  o[3] = __byte_perm(t2, t3, 0x7632);
}

// Per-thread constants of the item loop.
struct PackCtx {
  long long e1, e2, e3;  // ends of the interior, halo-row and halo-side ranges
  int cq_n;              // 16-byte chunks per pixel
  long long plane;       // D * H * W
};

__device__ __forceinline__ PackCtx pack_ctx(const ConvParams& p, const PackPlan& q) {
  PackCtx c;
  c.e1 = q.x_items;
  c.e2 = c.e1 + q.halo_row_items;
  c.e3 = c.e2 + q.halo_side_items;
  c.cq_n = p.C >> 4;
  c.plane = (long long)p.D * p.H * p.W;
  return c;
}

// Item g >= e1 of the pack: a zero chunk of the halo, or a weight chunk (g < e3 + w_items).
__device__ __forceinline__ void pack_rest_item(const ConvParams& p, const PackPlan& q,
                                               const PackCtx& c, long long g) {
  const long long e1 = c.e1, e2 = c.e2, e3 = c.e3;
  const int cq_n = c.cq_n;
  (void)q;
  if (g < e2) {
    // zero chunks of a halo row: halo planes first, then the halo rows of interior planes
    const long long gi = g - e1;
    const long long per_row = (long long)p.Wp * cq_n;
    const long long r = (gi / per_row);
    const long long chunk = gi - r * per_row;
    const long long halo_rows_per_image = (long long)p.Dp * p.Hp - (long long)p.D * p.H;
    const int n = (int)(r / halo_rows_per_image);
    long long rr = r - (long long)n * halo_rows_per_image;
    const long long front = (long long)p.pk_pd * p.Hp;
    int dp, hp;
    if (rr < front) {
      dp = (int)(rr / p.Hp);
      hp = (int)(rr % p.Hp);
    } else if (rr < 2 * front) {
      rr -= front;
      dp = p.pk_pd + p.D + (int)(rr / p.Hp);
      hp = (int)(rr % p.Hp);
    } else {
      rr -= 2 * front;
      const int side = 2 * p.pk_ph;
      const int kk = (int)(rr % side);
      dp = p.pk_pd + (int)(rr / side);
      hp = kk < p.pk_ph ? kk : p.H + kk;
    }
    *reinterpret_cast<uint4*>(p.xp + (((long long)n * p.Dp + dp) * p.Hp + hp) * p.Wp * p.C +
                              chunk * 16) = make_uint4(0u, 0u, 0u, 0u);
  } else if (g < e3) {
    // zero chunks of the W-halo pixels of interior rows
    const long long gi = g - e2;
    const int side = p.Wp - p.W;
    const long long per_row = (long long)side * cq_n;
    const long long row = gi / per_row;  // n*D*H + d*H + h
    const long long rem = gi - row * per_row;
    const int kk = (int)(rem / cq_n);
    const int cq = (int)(rem - (long long)kk * cq_n);
    const int wp = kk < p.pk_pw ? kk : p.W + kk;
    const int h = (int)(row % p.H);
    const int d = (int)((row / p.H) % p.D);
    const int n = (int)(row / ((long long)p.H * p.D));
    *reinterpret_cast<uint4*>(
        p.xp + ((((long long)n * p.Dp + d + p.pk_pd) * p.Hp + h + p.pk_ph) * p.Wp + wp) * p.C +
        cq * 16) = make_uint4(0u, 0u, 0u, 0u);
  } else {
    // weights: one item = one 16-byte chunk (16 e4m3 or 8 bfloat16 channels) of one tap
    const long long gw = g - e3;
    const int tap = (int)(gw % p.taps);
    const long long rest = gw / p.taps;
    const int cq = (int)(rest % cq_n);
    const int k = (int)(rest / cq_n);
    uint32_t v[4] = {0u, 0u, 0u, 0u};
    if (p.elem_bytes == 2) {
      const uint16_t* src = reinterpret_cast<const uint16_t*>(p.w) +
                            ((long long)k * (p.C >> 1) + cq * 8) * p.taps + tap;
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j >> 1] |= (uint32_t)__ldg(src + j * p.taps) << ((j & 1) * 16);
    } else {
      const uint8_t* src = p.w + ((long long)k * p.C + cq * 16) * p.taps + tap;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        v[j >> 2] |= (uint32_t)__ldg(src + j * p.taps) << ((j & 3) * 8);
    }
    uint4* dst =
        reinterpret_cast<uint4*>(p.wp + ((long long)k * p.taps + tap) * p.C + cq * 16);
    *dst = make_uint4(v[0], v[1], v[2], v[3]);
  }
}

// Item g of the pack (g < e3 + w_items).
__device__ __forceinline__ void pack_item(const ConvParams& p, const PackPlan& q,
                                          const PackCtx& c, long long g) {
  const long long e1 = c.e1;
  const int cq_n = c.cq_n;
  const long long plane = c.plane;
  if (g < e1 && q.copy) {
    // interior from a channels-last x: (chunk fastest, then pixel)
    const long long pix = g / cq_n;  // ((n*D + d)*H + h)*W + w
    const int cq = (int)(g - pix * cq_n);
    const int w = (int)(pix % p.W);
    const long long row = pix / p.W;
    const int h = (int)(row % p.H);
    const int d = (int)((row / p.H) % p.D);
    const int n = (int)(row / ((long long)p.H * p.D));
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.x + pix * p.C + cq * 16));
    *reinterpret_cast<uint4*>(
        p.xp + ((((long long)n * p.Dp + d + p.pk_pd) * p.Hp + h + p.pk_ph) * p.Wp + w + p.pk_pw) *
                   p.C + cq * 16) = v;
  } else if (g < e1 && p.elem_bytes == 2) {
    // interior, bfloat16: one item = 8 channels (one 16-byte chunk) x 8 pixels (W % 8 == 0), 2
    // pixels (W even) or 1; pixel group fastest, then chunk, then (n, d, h) row, or with the
    // chunk fastest (q.cfast)
    const int per_row = q.oct ? p.W / 8 : q.two ? p.W / 2 : p.W;
    int wi, cq;
    long long row;  // n*D*H + d*H + h
    if (q.cfast) {
      cq = (int)(g % cq_n);
      const long long rest = g / cq_n;
      wi = (int)(rest % per_row);
      row = rest / per_row;
    } else {
      wi = (int)(g % per_row);
      const long long rest = g / per_row;
      cq = (int)(rest % cq_n);
      row = rest / cq_n;
    }
    const int h = (int)(row % p.H);
    const int d = (int)((row / p.H) % p.D);
    const int n = (int)(row / ((long long)p.H * p.D));
    const int c_el = p.C >> 1;
    const uint16_t* src = reinterpret_cast<const uint16_t*>(p.x) +
                          ((long long)n * c_el + cq * 8) * plane + ((long long)d * p.H + h) * p.W;
    uint8_t* dst_row = p.xp + ((((long long)n * p.Dp + d + p.pk_pd) * p.Hp + h + p.pk_ph) *
                                   p.Wp + p.pk_pw) * p.C + cq * 16;
    if (q.oct) {
      // a[c]: pixels 8wi..8wi+7 of channel c, two to a word (the even pixel in the low half);
      // pixel 2k+j's channel pair (2m, 2m+1) is half j of word k of a[2m] and of a[2m+1]
      uint4 a[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) a[c] = __ldg(reinterpret_cast<const uint4*>(src + c * plane) + wi);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t lo[4], hi[4];  // channel pairs of pixel 8wi + 2k and of pixel 8wi + 2k + 1
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint32_t e = k == 0 ? a[2 * m].x : k == 1 ? a[2 * m].y : k == 2 ? a[2 * m].z : a[2 * m].w;
          const uint32_t o = k == 0   ? a[2 * m + 1].x
                             : k == 1 ? a[2 * m + 1].y
                             : k == 2 ? a[2 * m + 1].z
                                      : a[2 * m + 1].w;
          lo[m] = __byte_perm(e, o, 0x5410);
          hi[m] = __byte_perm(e, o, 0x7632);
        }
        *reinterpret_cast<uint4*>(dst_row + (long long)(8 * wi + 2 * k) * p.C) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<uint4*>(dst_row + (long long)(8 * wi + 2 * k + 1) * p.C) =
            make_uint4(hi[0], hi[1], hi[2], hi[3]);
      }
    } else if (q.two) {
      uint32_t v[8];  // v[c]: pixels 2wi (low half) and 2wi+1 (high half) of channel c
#pragma unroll
      for (int j = 0; j < 8; ++j)
        v[j] = __ldg(reinterpret_cast<const uint32_t*>(src + j * plane) + wi);
      uint32_t lo[4], hi[4];  // channel pairs (2k, 2k+1) of pixel 2wi and of pixel 2wi+1
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        lo[k] = __byte_perm(v[2 * k], v[2 * k + 1], 0x5410);
        hi[k] = __byte_perm(v[2 * k], v[2 * k + 1], 0x7632);
      }
      *reinterpret_cast<uint4*>(dst_row + (long long)(2 * wi) * p.C) =
          make_uint4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<uint4*>(dst_row + (long long)(2 * wi + 1) * p.C) =
          make_uint4(hi[0], hi[1], hi[2], hi[3]);
    } else {
      uint32_t v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        v[k] = (uint32_t)__ldg(src + (2 * k) * plane + wi) |
               ((uint32_t)__ldg(src + (2 * k + 1) * plane + wi) << 16);
      *reinterpret_cast<uint4*>(dst_row + (long long)wi * p.C) = make_uint4(v[0], v[1], v[2], v[3]);
    }
  } else if (g < e1) {
    // interior: (pixel group fastest, then channel chunk, then (n, d, h) row), or with the
    // channel chunk fastest (q.cfast)
    const int per_row = q.hex ? p.W / 16 : q.quad ? p.W / 4 : p.W;
    int wi, cq;
    long long row;  // n*D*H + d*H + h
    if (q.cfast) {
      cq = (int)(g % cq_n);
      const long long rest = g / cq_n;
      wi = (int)(rest % per_row);
      row = rest / per_row;
    } else {
      wi = (int)(g % per_row);
      const long long rest = g / per_row;
      cq = (int)(rest % cq_n);
      row = rest / cq_n;
    }
    const int h = (int)(row % p.H);
    const int d = (int)((row / p.H) % p.D);
    const int n = (int)(row / ((long long)p.H * p.D));
    const uint8_t* src = p.x + ((long long)n * p.C + cq * 16) * plane +
                         ((long long)d * p.H + h) * p.W;
    uint8_t* dst_row = p.xp + ((((long long)n * p.Dp + d + p.pk_pd) * p.Hp + h + p.pk_ph) *
                                   p.Wp + p.pk_pw) * p.C + cq * 16;
    if (q.hex) {
      // 16 channels x 16 pixels: one 16-byte load per channel, then four 4-pixel groups through
      // the same 4x4 byte transposes as the quad items
      uint4 u[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        u[j] = __ldg(reinterpret_cast<const uint4*>(src + j * plane) + wi);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          v[j] = k == 0 ? u[j].x : k == 1 ? u[j].y : k == 2 ? u[j].z : u[j].w;
        uint32_t o[4][4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t t[4];
          transpose4x4(v + 4 * b, t);
#pragma unroll
          for (int j = 0; j < 4; ++j) o[j][b] = t[j];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(dst_row + (long long)(16 * wi + 4 * k + j) * p.C) =
              make_uint4(o[j][0], o[j][1], o[j][2], o[j][3]);
      }
    } else if (q.quad) {
      uint32_t v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        v[j] = __ldg(reinterpret_cast<const uint32_t*>(src + j * plane) + wi);
      uint32_t o[4][4];  // o[pixel][word of 4 channels]
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        uint32_t t[4];
        transpose4x4(v + 4 * b, t);
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j][b] = t[j];
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(dst_row + (long long)(4 * wi + j) * p.C) =
            make_uint4(o[j][0], o[j][1], o[j][2], o[j][3]);
    } else {
      uint32_t v[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int j = 0; j < 16; ++j)
        v[j >> 2] |= (uint32_t)__ldg(src + j * plane + wi) << ((j & 3) * 8);
      *reinterpret_cast<uint4*>(dst_row + (long long)wi * p.C) = make_uint4(v[0], v[1], v[2], v[3]);
    }
  } else {
    pack_rest_item(p, q, c, g);
  }
}

// Weight tile wb of the re-layout KCTRS -> K x taps x C: filter k and the w_group 16-byte channel
// chunks from cq0 on. Their source is one contiguous run of nq * 16 * taps bytes (channel-major,
// taps innermost), copied into `sm` with 16-byte loads; then each thread gathers one 16-byte chunk
// of one tap (16 e4m3 or 8 bfloat16 channels, taps bytes apart in shared memory) and stores it
// with one 16-byte store. Every thread of the block must call it (it synchronises the block).
__device__ __forceinline__ void pack_w_tile(const ConvParams& p, const PackPlan& q, long long wb,
                                            uint8_t* sm) {
  const int cq_n = p.C >> 4;
  const int ng = (cq_n + q.w_group - 1) / q.w_group;
  const int k = (int)(wb / ng);
  const int cq0 = (int)(wb - (long long)k * ng) * q.w_group;
  const int nq = min(q.w_group, cq_n - cq0);
  const int taps = p.taps;
  const uint8_t* src = p.w + ((long long)k * p.C + (long long)cq0 * 16) * taps;
  const int vecs = nq * taps;  // 16-byte vectors of the run
  for (int v = threadIdx.x; v < vecs; v += blockDim.x)
    reinterpret_cast<uint4*>(sm)[v] = __ldg(reinterpret_cast<const uint4*>(src) + v);
  __syncthreads();
  for (int t = threadIdx.x; t < vecs; t += blockDim.x) {
    const int cl = t / taps, tap = t - cl * taps;  // chunk within the tile, tap
    uint32_t v[4] = {0u, 0u, 0u, 0u};
    if (p.elem_bytes == 2) {
      const uint16_t* s16 = reinterpret_cast<const uint16_t*>(sm) + (cl * 8) * taps + tap;
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j >> 1] |= (uint32_t)s16[j * taps] << ((j & 1) * 16);
    } else {
      const uint8_t* s8 = sm + (cl * 16) * taps + tap;
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j >> 2] |= (uint32_t)s8[j * taps] << ((j & 3) * 8);
    }
    *reinterpret_cast<uint4*>(p.wp + ((long long)k * taps + tap) * p.C +
                              (long long)(cq0 + cl) * 16) = make_uint4(v[0], v[1], v[2], v[3]);
  }
}

}  // namespace c3d
