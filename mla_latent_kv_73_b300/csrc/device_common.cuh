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

// cos/sin of the RoPE angle pos * theta_i, theta_i = base^(-2i/d_r).
// rope_turns holds theta_i / (2 pi) as a 64-bit binary fraction of a turn
// (built on the host in extended precision). The integer product
// pos * rope_turns, taken modulo 2^64, is then exactly the fractional part of
// the angle in turns, with no range reduction and no fp64 arithmetic (B300's
// fp64 rate is low). Its top 32 bits, read as a signed number, are the angle
// in [-1/2, 1/2) turns; sincospif evaluates sin/cos of pi times twice that.
// The representation error of theta_i / (2 pi) is at most 2^-65 turns, so
// the product is good to about 2^-48 turns at positions up to 2^17; the fp32
// argument of sincospif then keeps 24 bits of it, as a directly reduced fp32
// angle would.
__device__ __forceinline__ void rope_cos_sin(int pos, uint64_t rope_turns, float* c, float* s) {
  const uint64_t f = static_cast<uint64_t>(static_cast<uint32_t>(pos)) * rope_turns;
  const int32_t hi = static_cast<int32_t>(static_cast<uint32_t>(f >> 32));
  sincospif(static_cast<float>(hi) * 0x1p-31f, s, c);
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
