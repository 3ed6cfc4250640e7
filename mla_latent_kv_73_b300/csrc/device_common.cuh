// Device helpers shared by the libmla kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "mla_internal.h"

namespace mla {

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// cos/sin of pos * base^(-2i/d) with the angle formed in fp64, so that
// positions up to 2^31 keep their accuracy. CUDA's own sincos is called.
__device__ __forceinline__ void rope_cos_sin(int pos, int i, int d, float base, float* c,
                                             float* s) {
  const double inv_freq = pow(static_cast<double>(base), -2.0 * i / d);
  double sd, cd;
  sincos(static_cast<double>(pos) * inv_freq, &sd, &cd);
  *c = static_cast<float>(cd);
  *s = static_cast<float>(sd);
}

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

// The CTA that owns flat work item x when N items are split over C CTAs
// as [c*N/C, (c+1)*N/C).
__device__ __forceinline__ int cta_of_item(long long x, long long N, int C) {
  return static_cast<int>(((x + 1) * C - 1) / N);
}
__device__ __forceinline__ long long range_begin(int c, long long N, int C) {
  return (static_cast<long long>(c) * N) / C;
}

}  // namespace mla
