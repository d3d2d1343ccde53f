// pack.cu -- operand re-layout in front of the implicit GEMM, and the split-K reduction behind it.
//
// The GEMM view orders K_gemm as (tap, channel) with the channel innermost, so that one row of the
// A tile for one tap is C contiguous bytes of one input pixel. The caller's x is NCDHW (channel
// outermost), so it is copied once per run into a channels-last buffer. For the TMA im2col route
// the copy is plain NDHWC (the TMA unit zero-fills taps outside the volume); for the cp.async
// gather route it carries an explicit zero halo of `pad` pixels on every spatial side, so that an
// A-tile row needs no bounds test, only the padded-row test (row < npq). The weights are re-laid
// from KCTRS to K x taps x C to match.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "conv_common.cuh"

namespace c3d {

// One thread writes 16 channels (16 bytes) of one padded pixel, or 16 channels of one tap of one
// filter. Pixels run fastest across threads so that each of the 16 byte loads of a warp is a
// contiguous run along W of the NCDHW input.
__global__ void __launch_bounds__(256) pack_kernel(ConvParams p, long long x_items,
                                                   long long w_items) {
  const long long total = x_items + w_items;
  const int cq_n = p.C >> 4;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x) {
    uint32_t v[4] = {0u, 0u, 0u, 0u};
    if (g < x_items) {
      const int wpos = (int)(g % p.Wp);
      long long rest = g / p.Wp;
      const int cq = (int)(rest % cq_n);
      const long long prow = rest / cq_n;         // (n, dp, hp) of the padded volume
      const int hp = (int)(prow % p.Hp);
      const int dp = (int)((prow / p.Hp) % p.Dp);
      const int n = (int)(prow / ((long long)p.Hp * p.Dp));
      const int d = dp - p.pk_pd, h = hp - p.pk_ph, w = wpos - p.pk_pw;
      if (d >= 0 && d < p.D && h >= 0 && h < p.H && w >= 0 && w < p.W) {
        const long long plane = (long long)p.D * p.H * p.W;
        const uint8_t* src =
            p.x + ((long long)n * p.C + cq * 16) * plane + ((long long)d * p.H + h) * p.W + w;
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j >> 2] |= (uint32_t)__ldg(src + j * plane) << ((j & 3) * 8);
      }
      uint4* dst = reinterpret_cast<uint4*>(p.xp + (prow * p.Wp + wpos) * p.C + cq * 16);
      *dst = make_uint4(v[0], v[1], v[2], v[3]);
    } else {
      const long long gw = g - x_items;
      const int tap = (int)(gw % p.taps);
      const long long rest = gw / p.taps;
      const int cq = (int)(rest % cq_n);
      const int k = (int)(rest / cq_n);
      const uint8_t* src = p.w + ((long long)k * p.C + cq * 16) * p.taps + tap;
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j >> 2] |= (uint32_t)__ldg(src + j * p.taps) << ((j & 3) * 8);
      uint4* dst =
          reinterpret_cast<uint4*>(p.wp + ((long long)k * p.taps + tap) * p.C + cq * 16);
      *dst = make_uint4(v[0], v[1], v[2], v[3]);
    }
  }
}

cudaError_t launch_pack(const ConvParams& p, cudaStream_t stream) {
  const long long x_items = (long long)p.N * p.Dp * p.Hp * p.Wp * (p.C / 16);
  const long long w_items = (long long)p.K * p.taps * (p.C / 16);
  const long long total = x_items + w_items;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)sms * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  pack_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, x_items, w_items);
  return cudaGetLastError();
}

// Split-K reduction: y = bf16(scale * sum_{split = 0..splits-1} partial[split]) in ascending split
// order, so the result is bitwise reproducible for a fixed plan. One thread per (tile, column,
// row); the stores carry the same guards as the main epilogue (real output row, col < K).
template <bool kRowChk>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(ConvParams p) {
  const long long per_tile = (long long)p.block_n * p.block_m;
  const long long total = (long long)p.m_tiles * p.n_tiles * per_tile;
  const float scale = __ldg(p.scale_x) * __ldg(p.scale_w);
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(g % p.block_m);
    const int col_l = (int)((g / p.block_m) % p.block_n);
    const long long tile = g / per_tile;
    const int n_tile = (int)(tile % p.n_tiles);
    const int m_tile = (int)(tile / p.n_tiles);
    const int col = n_tile * p.block_n + col_l;
    if (col >= p.K) continue;
    const RowDest dst = row_dest(p, m_tile, row);
    if (kRowChk && !dst.valid) continue;
    const float* src = p.partials + ((tile * p.splits) * p.block_n + col_l) * p.block_m + row;
    float acc = 0.0f;
    for (int s = 0; s < p.splits; ++s) acc += __ldcg(src + (long long)s * per_tile);
    const __nv_bfloat16 b = __float2bfloat16_rn(acc * scale);
    p.y[dst.y_off + (long long)col * p.dhw] = *reinterpret_cast<const uint16_t*>(&b);
  }
}

cudaError_t launch_splitk_reduce(const ConvParams& p, bool row_chk, cudaStream_t stream) {
  const long long total = (long long)p.m_tiles * p.n_tiles * p.block_n * p.block_m;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)sms * 16;
  if (blocks > cap) blocks = cap;
  if (row_chk)
    splitk_reduce_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(p);
  else
    splitk_reduce_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace c3d
