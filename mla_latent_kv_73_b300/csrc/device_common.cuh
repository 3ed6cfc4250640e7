// Device helpers shared by the libmla kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
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
template <>
__device__ __forceinline__ __half from_f32<__half>(float v) {
  return __float2half_rn(v);
}

// cos/sin of pos * inv_freq, where inv_freq = base^(-2i/d_r) comes from a
// table built on the host in fp64. The angle is formed in fp64 and reduced
// to [-pi, pi] with one fused multiply-add against 2*pi (Cody-Waite style,
// one constant). The reduced angle is good to about 1e-11 rad at positions
// up to 2^17, and to about 1e-6 rad at 2^31. CUDA's fp32 sincosf then
// evaluates it. Each angle costs 4 fp64 operations, which matters because
// B300's fp64 rate is low.
__device__ __forceinline__ void rope_cos_sin(int pos, double inv_freq, float* c, float* s) {
  const double two_pi = 6.283185307179586;
  const double a = static_cast<double>(pos) * inv_freq;
  const double k = rint(a * 0.15915494309189535);
  const float r = static_cast<float>(fma(-k, two_pi, a));
  sincosf(r, s, c);
}

// 16-byte vector loads of T, widened to fp32.
template <typename T>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int N = 4;
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
};

template <typename T>
__device__ __forceinline__ void load_vec(const T* p, float (&v)[Vec<T>::N]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(p);
  if constexpr (sizeof(T) == 4) {
    v[0] = __uint_as_float(raw.x);
    v[1] = __uint_as_float(raw.y);
    v[2] = __uint_as_float(raw.z);
    v[3] = __uint_as_float(raw.w);
  } else {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

}  // namespace mla
