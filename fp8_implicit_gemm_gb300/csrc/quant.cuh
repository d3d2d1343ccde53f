// quant.cuh -- device helpers of the per-tensor e4m3 quantiser, shared by the standalone cast
// (quant.cu) and the pack's quantise-and-transpose of x (pack.cu).
#pragma once
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "conv3d_fp8_internal.h"

namespace c3d {

// 16 bytes of source as fp32 values (4 fp32 or 8 bfloat16 elements)
__device__ __forceinline__ void load16_f32(const uint8_t* p, float (&v)[4]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  v[0] = a.x;
  v[1] = a.y;
  v[2] = a.z;
  v[3] = a.w;
}
__device__ __forceinline__ void load16_bf16(const uint8_t* p, float (&v)[8]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);  // low half: the element at the lower address
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float src_value(const void* src, int type, long long i) {
  if (type == kSrcF32) return __ldg(static_cast<const float*>(src) + i);
  const uint16_t b = __ldg(static_cast<const uint16_t*>(src) + i);
  return __uint_as_float((uint32_t)b << 16);
}

__device__ __forceinline__ float scale_from_amax(unsigned amax_bits) {
  const float amax = __uint_as_float(amax_bits);
  return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

// Four values -> four e4m3 codes (the first in the lowest byte). The clamp to +-448 is the
// conversion's own saturation: a quotient above 448 in magnitude rounds to 448 or to the first
// magnitude past it, which saturates to 448 -- the code of the clamped value either way.
__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float s) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s)),
                                               __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(c, s), __fdiv_rn(d, s)),
                                               __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}

}  // namespace c3d
