// a0: repack the weights once at load time.
//
// Source: "Multi-head Latent Attention: the KV cache, compressed", section
// "Store the archive, not the files". Folding the up-projections is done once,
// when the model loads, and never per step. Here that means W_uk is laid out
// per head for the query-side fold, W_uv per head for the output-side fold,
// and [W_dkv | W_kr] one output column per row for the compress-and-append
// kernel. The packing only copies and transposes. It does no arithmetic.
// (The RoPE inverse-frequency table is filled on the host.)
#include "device_common.cuh"

namespace mla {
namespace {

// Wp[col][k] = W_dkv[k][col] for col < d_c;
// Wp[d_c + 2i + e][k] = W_kr[k][i + e*d_r/2] (the rotary pairs are interleaved).
template <typename T>
__global__ void pack_dkvr_kernel(const T* __restrict__ W_dkv, const T* __restrict__ W_kr,
                                 T* __restrict__ Wp, int d_model, int d_c, int d_r) {
  __shared__ T tile[32][33];
  const int R = d_c + d_r;
  const int k0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  // read a 32x32 tile: rows k, columns col (logical packed column)
  for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
    const int k = k0 + dy, col = c0 + threadIdx.x;
    T v = from_f32<T>(0.f);
    if (k < d_model && col < R) {
      if (col < d_c) {
        v = W_dkv[static_cast<size_t>(k) * d_c + col];
      } else {
        const int j = col - d_c, i = j >> 1, e = j & 1;
        v = W_kr[static_cast<size_t>(k) * d_r + i + e * (d_r / 2)];
      }
    }
    tile[dy][threadIdx.x] = v;
  }
  __syncthreads();
  for (int dy = threadIdx.y; dy < 32; dy += blockDim.y) {
    const int col = c0 + dy, k = k0 + threadIdx.x;
    if (col < R && k < d_model) Wp[static_cast<size_t>(col) * d_model + k] = tile[threadIdx.x][dy];
  }
}

// W [d_c, n_h*d] (row-major) -> Wp [n_h][d_c][d]
template <typename T>
__global__ void pack_per_head_kernel(const T* __restrict__ W, T* __restrict__ Wp, int d_c,
                                     int n_h, int d) {
  const size_t total = static_cast<size_t>(n_h) * d_c * d;
  for (size_t o = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; o < total;
       o += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(o % d);
    const size_t t = o / d;
    const int c = static_cast<int>(t % d_c);
    const int h = static_cast<int>(t / d_c);
    Wp[o] = W[static_cast<size_t>(c) * n_h * d + static_cast<size_t>(h) * d + j];
  }
}

// W [d_c, n_h*d] (row-major) -> Wp [n_h][d][d_c]: each output column contiguous
template <typename T>
__global__ void pack_per_head_t_kernel(const T* __restrict__ W, T* __restrict__ Wp, int d_c,
                                       int n_h, int d) {
  const size_t total = static_cast<size_t>(n_h) * d_c * d;
  for (size_t o = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; o < total;
       o += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(o % d_c);
    const size_t t = o / d_c;
    const int j = static_cast<int>(t % d);
    const int h = static_cast<int>(t / d);
    Wp[o] = W[static_cast<size_t>(c) * n_h * d + static_cast<size_t>(h) * d + j];
  }
}

template <typename T>
cudaError_t pack_all(const Shape& s, const void* W_dkv, const void* W_kr, const void* W_uk,
                     const void* W_uv, Weights* w, cudaStream_t st) {
  const int R = s.R();
  dim3 blk(32, 8), grd((s.d_model + 31) / 32, (R + 31) / 32);
  pack_dkvr_kernel<T><<<grd, blk, 0, st>>>(static_cast<const T*>(W_dkv),
                                          static_cast<const T*>(W_kr), static_cast<T*>(w->w_dkvr),
                                          s.d_model, s.d_c, s.d_r);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  pack_per_head_kernel<T><<<1024, 256, 0, st>>>(static_cast<const T*>(W_uk),
                                                static_cast<T*>(w->w_uk), s.d_c, s.n_h, s.d_nope);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  pack_per_head_t_kernel<T><<<1024, 256, 0, st>>>(static_cast<const T*>(W_uv),
                                                  static_cast<T*>(w->w_uv), s.d_c, s.n_h, s.d_v);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack_weights(const Shape& s, mla_dtype dt, const void* W_dkv, const void* W_kr,
                                const void* W_uk, const void* W_uv, Weights* w, cudaStream_t st) {
  if (dt == MLA_F32) return pack_all<float>(s, W_dkv, W_kr, W_uk, W_uv, w, st);
  return pack_all<__nv_bfloat16>(s, W_dkv, W_kr, W_uk, W_uv, w, st);
}

}  // namespace mla
