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

#include "pack_items.cuh"

namespace c3d {

__global__ void __launch_bounds__(256) pack_kernel(ConvParams p, PackPlan q) {
  pdl_launch_dependents();  // the implicit GEMM may start its prologue while the pack runs
  const PackCtx c = pack_ctx(p, q);
  const long long total = c.e3 + q.w_items;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x)
    pack_item(p, q, c, g);
}

cudaError_t launch_pack(const ConvParams& p, cudaStream_t stream) {
  const PackPlan q = pack_plan(p);
  const long long total = q.x_items + q.halo_row_items + q.halo_side_items + q.w_items;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)sms * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  pack_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, q);
  return cudaGetLastError();
}

// Split-K reduction of the split tiles (full_tiles..m_tiles*n_tiles-1):
// y = bf16(scale * sum_{split = 0..splits-1} partial[split]) in ascending split order, so the
// result is bitwise reproducible for a fixed plan. One thread per (tile, column, row); the stores
// carry the same guards as the main epilogue (real output row, col < K).
template <bool kRowChk>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(ConvParams p) {
  const long long per_tile = (long long)p.block_n * p.block_m;
  const long long total = ((long long)p.m_tiles * p.n_tiles - p.full_tiles) * per_tile;
  pdl_wait_primary();  // the partials of the implicit GEMM, complete and visible
  const float scale = __ldg(p.scale_x) * __ldg(p.scale_w);
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(g % p.block_m);
    const int col_l = (int)((g / p.block_m) % p.block_n);
    const long long t = g / per_tile;  // index among the split tiles
    const long long tile = p.full_tiles + t;
    const int n_tile = (int)(tile % p.n_tiles);
    const int m_tile = (int)(tile / p.n_tiles);
    const int col = n_tile * p.block_n + col_l;
    if (col >= p.K) continue;
    const RowDest dst = row_dest(p, m_tile, row);
    if (kRowChk && !dst.valid) continue;
    const float* src = p.partials + ((t * p.splits) * p.block_n + col_l) * p.block_m + row;
    // eight loads in flight at a time; the additions stay in ascending split order
    float acc = 0.0f;
    int s = 0;
    for (; s + 8 <= p.splits; s += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __ldcg(src + (long long)(s + j) * per_tile);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc += v[j];
    }
    for (; s < p.splits; ++s) acc += __ldcg(src + (long long)s * per_tile);
    const __nv_bfloat16 b = __float2bfloat16_rn(acc * scale);
    p.y[dst.y_off + (long long)col * p.dhw] = *reinterpret_cast<const uint16_t*>(&b);
  }
}

cudaError_t launch_splitk_reduce(const ConvParams& p, bool row_chk, cudaStream_t stream) {
  const long long total =
      ((long long)p.m_tiles * p.n_tiles - p.full_tiles) * p.block_n * p.block_m;
  if (total <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)sms * 16;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return row_chk ? cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<true>, p)
                 : cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<false>, p);
}

}  // namespace c3d
