// fp8 (e4m3) latent cache: the row quantiser.
//
//   scale_t = max_k |row_t[k]| / 448      (1 for a row of zeros)
//   code_t[k] = e4m3(row_t[k] / scale_t)  (round to nearest, ties to even)
//   cache[page_table[b][pos_t / bs]][pos_t % bs][:] = code_t, row_scale[...] = scale_t
//
// Source: "Multi-head Latent Attention and KV Cache Compression", section
// "Moving a trained MHA model over": quantisation can be stacked on top of
// the latent cache, and its error then passes through the up-projections
// into every head's keys and values. The page fixes neither the format nor
// the scale granularity. The reading taken here: e4m3 in the "fn" variant
// (bias 7, 3 mantissa bits, largest finite value 448, no infinities) with
// one fp32 scale per cache row, chosen so that the row's largest element
// becomes +-448. The scale and the division are computed in fp32 with
// correct rounding, and the conversion saturates (a quotient a rounding step
// above 448 becomes 448).
//
// One warp per token: each lane holds every 32nd element of the row, the
// warp reduces |x| to the row maximum with shuffles, then writes the codes
// (consecutive lanes, consecutive bytes) and lane 0 the scale.
#include <cuda_fp8.h>

#include "device_common.cuh"

namespace mla {
namespace {

constexpr int QZ_WARPS = 8;
constexpr int QZ_MAX_PER_LANE = 32;  // R <= 1024

__global__ void __launch_bounds__(QZ_WARPS * 32)
quantize_rows_fp8_kernel(Shape s, const float* __restrict__ rows,
                         const int32_t* __restrict__ seq_idx, const int32_t* __restrict__ pos,
                         const int32_t* __restrict__ page_table, int B, int max_blocks,
                         int num_blocks, int T, uint8_t* __restrict__ codes,
                         float* __restrict__ row_scale, uint32_t* err) {
  const int lane = threadIdx.x % 32;
  const int t = blockIdx.x * QZ_WARPS + threadIdx.x / 32;
  if (t >= T) return;
  const int R = s.R();
  const int b = seq_idx[t], p = pos[t];
  if (b < 0 || b >= B || p < 0 || p / s.bs >= max_blocks) {
    if (lane == 0) set_error(err, MLA_DEVERR_APPEND_INDEX);
    return;
  }
  const int page = page_table[static_cast<size_t>(b) * max_blocks + p / s.bs];
  if (page < 0 || page >= num_blocks) {
    if (lane == 0) set_error(err, MLA_DEVERR_PAGE_RANGE);
    return;
  }
  const long long row = static_cast<long long>(page) * s.bs + p % s.bs;
  const float* src = rows + static_cast<size_t>(t) * R;
  float v[QZ_MAX_PER_LANE];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < QZ_MAX_PER_LANE; ++i) {
    const int k = lane + 32 * i;
    v[i] = k < R ? src[k] : 0.f;
    amax = fmaxf(amax, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.f ? amax / 448.f : 1.f;
  uint8_t* dst = codes + row * R;
#pragma unroll
  for (int i = 0; i < QZ_MAX_PER_LANE; ++i) {
    const int k = lane + 32 * i;
    if (k < R) dst[k] = __nv_cvt_float_to_fp8(v[i] / scale, __NV_SATFINITE, __NV_E4M3);
  }
  if (lane == 0) row_scale[row] = scale;
}

}  // namespace

cudaError_t launch_quantize_rows_fp8(const Shape& s, const float* rows, const int32_t* seq_idx,
                                     const int32_t* pos, const int32_t* page_table, int B,
                                     int max_blocks, uint8_t* codes, float* row_scale,
                                     int num_blocks, int T, uint32_t* err, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (s.R() > 32 * QZ_MAX_PER_LANE) return cudaErrorInvalidValue;
  const int grid = (T + QZ_WARPS - 1) / QZ_WARPS;
  quantize_rows_fp8_kernel<<<grid, QZ_WARPS * 32, 0, st>>>(s, rows, seq_idx, pos, page_table, B,
                                                           max_blocks, num_blocks, T, codes,
                                                           row_scale, err);
  return cudaGetLastError();
}

}  // namespace mla
