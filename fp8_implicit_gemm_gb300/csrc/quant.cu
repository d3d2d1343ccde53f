// quant.cu -- per-tensor e4m3 quantiser on the GPU: the producer of the e4m3 bytes and of the
// per-tensor scale that the implicit GEMM consumes ("fp8cast" on the subject page, "[Fix] conv3d
// fp8: guard padded M rows in the epilogue store", section "Problem").
//
//   amax = max |v|,  s = fp32(amax / 448) (1 when amax == 0),
//   q = e4m3_rne(clamp(fp32(v / s), +-448))
//
// Three launches, no host synchronisation: an amax reduction into a device word (the bit pattern
// of a non-negative float orders like the float, so an integer max is the float max), the cast
// (IEEE fp32 division, then the hardware's satfinite round-to-nearest-even e4m3 conversion), and
// a one-thread finalisation that turns the amax into the scale. The cast of x can instead be
// fused into the pack of a run (pack.cu, x_src_type != 0), which reads the finalised scale.
// NaN inputs are not supported (the reduction would carry them into the scale).
#include <cuda_runtime.h>

#include "conv3d_fp8_internal.h"
#include "quant.cuh"

namespace c3d {

constexpr int kQuantThreads = 256;

// Each thread takes 64 bytes of source per step (4 independent 16-byte loads), so that enough
// bytes are in flight to run at the memory's bandwidth.
constexpr int kQuantVecs = 4;

__global__ void __launch_bounds__(kQuantThreads) amax_kernel(const void* src, int type,
                                                             long long n, unsigned* amax_bits) {
  const int per_vec = type == kSrcF32 ? 4 : 8;  // elements in 16 bytes
  const long long nblk = n / (per_vec * kQuantVecs);
  const uint8_t* base = static_cast<const uint8_t*>(src);
  float m = 0.0f;
  const long long stride = (long long)gridDim.x * blockDim.x;
  // The sweep runs from the end of the source to its start: the pass that follows (the cast, or
  // the quantising pack) reads from the start, which is then the part still in L2.
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nblk; i += stride) {
    const uint8_t* p = base + (nblk - 1 - i) * 16 * kQuantVecs;
    if (type == kSrcF32) {
      float v[kQuantVecs][4];
#pragma unroll
      for (int k = 0; k < kQuantVecs; ++k) load16_f32(p + 16 * k, v[k]);
#pragma unroll
      for (int k = 0; k < kQuantVecs; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j) m = fmaxf(m, fabsf(v[k][j]));
    } else {
      float v[kQuantVecs][8];
#pragma unroll
      for (int k = 0; k < kQuantVecs; ++k) load16_bf16(p + 16 * k, v[k]);
#pragma unroll
      for (int k = 0; k < kQuantVecs; ++k)
#pragma unroll
        for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[k][j]));
    }
  }
  for (long long i = nblk * per_vec * kQuantVecs + blockIdx.x * (long long)blockDim.x +
                     threadIdx.x;
       i < n; i += stride)
    m = fmaxf(m, fabsf(src_value(src, type, i)));
  unsigned bits = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m));
  __shared__ unsigned warp_max[kQuantThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = bits;
  __syncthreads();
  if (threadIdx.x < 32) {
    bits = threadIdx.x < kQuantThreads / 32 ? warp_max[threadIdx.x] : 0u;
    bits = __reduce_max_sync(0xFFFFFFFFu, bits);
    if (threadIdx.x == 0) atomicMax(amax_bits, bits);
  }
}

// One step of a thread: 64 bytes of source = 16 fp32 or 32 bfloat16 values -> 16 or 32 codes.
__global__ void __launch_bounds__(kQuantThreads) quant_cast_kernel(const void* src, int type,
                                                                   long long n, uint8_t* dst,
                                                                   const unsigned* amax_bits) {
  const float s = scale_from_amax(*amax_bits);
  const int per_step = type == kSrcF32 ? 16 : 32;  // values in 64 bytes of source
  const long long nstep = n / per_step;
  const uint8_t* base = static_cast<const uint8_t*>(src);
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nstep; i += stride) {
    const uint8_t* p = base + i * 64;
    if (type == kSrcF32) {
      float v[4][4];
#pragma unroll
      for (int k = 0; k < 4; ++k) load16_f32(p + 16 * k, v[k]);
      uint4 o;
      o.x = quant4(v[0][0], v[0][1], v[0][2], v[0][3], s);
      o.y = quant4(v[1][0], v[1][1], v[1][2], v[1][3], s);
      o.z = quant4(v[2][0], v[2][1], v[2][2], v[2][3], s);
      o.w = quant4(v[3][0], v[3][1], v[3][2], v[3][3], s);
      *reinterpret_cast<uint4*>(dst + i * 16) = o;
    } else {
      float v[4][8];
#pragma unroll
      for (int k = 0; k < 4; ++k) load16_bf16(p + 16 * k, v[k]);
      uint4 o[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        o[h].x = quant4(v[2 * h][0], v[2 * h][1], v[2 * h][2], v[2 * h][3], s);
        o[h].y = quant4(v[2 * h][4], v[2 * h][5], v[2 * h][6], v[2 * h][7], s);
        o[h].z = quant4(v[2 * h + 1][0], v[2 * h + 1][1], v[2 * h + 1][2], v[2 * h + 1][3], s);
        o[h].w = quant4(v[2 * h + 1][4], v[2 * h + 1][5], v[2 * h + 1][6], v[2 * h + 1][7], s);
      }
      *reinterpret_cast<uint4*>(dst + i * 32) = o[0];
      *reinterpret_cast<uint4*>(dst + i * 32 + 16) = o[1];
    }
  }
  for (long long i = nstep * per_step + blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += stride)
    dst[i] = (uint8_t)(quant4(src_value(src, type, i), 0.0f, 0.0f, 0.0f, s) & 0xFFu);
}

// scale_out[0] (and scale_copy[0], if given) = the scale of the reduced amax
__global__ void quant_finalize_kernel(const unsigned* amax_bits, float* scale_out,
                                      float* scale_copy) {
  const float s = scale_from_amax(*amax_bits);
  *scale_out = s;
  if (scale_copy) *scale_copy = s;
}

static int quant_blocks(long long work) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long b = (work + kQuantThreads - 1) / kQuantThreads;
  const long long cap = (long long)(sms > 0 ? sms : 1) * 16;
  if (b > cap) b = cap;
  return b < 1 ? 1 : (int)b;
}

cudaError_t launch_amax(const void* src, int type, long long n, unsigned* amax_bits,
                        cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  const long long steps = n / ((type == kSrcF32 ? 4 : 8) * kQuantVecs);
  amax_kernel<<<quant_blocks(steps > 0 ? steps : 1), kQuantThreads, 0, stream>>>(src, type, n,
                                                                                amax_bits);
  return cudaGetLastError();
}

cudaError_t launch_quant_cast(const void* src, int type, long long n, uint8_t* dst,
                              const unsigned* amax_bits, cudaStream_t stream) {
  const long long steps = n / (type == kSrcF32 ? 16 : 32);
  quant_cast_kernel<<<quant_blocks(steps > 0 ? steps : 1), kQuantThreads, 0, stream>>>(
      src, type, n, dst, amax_bits);
  return cudaGetLastError();
}

cudaError_t launch_quant_finalize(const unsigned* amax_bits, float* scale_out, float* scale_copy,
                                  cudaStream_t stream) {
  quant_finalize_kernel<<<1, 1, 0, stream>>>(amax_bits, scale_out, scale_copy);
  return cudaGetLastError();
}

}  // namespace c3d
