// a1: compress new tokens and append them to the paged latent cache.
//
//   row_t = [ x_t W_dkv | RoPE(x_t W_kr, pos_t) ]
//   cache[page_table[b][pos_t / bs]][pos_t % bs][:] = round(row_t)
//
// Sources: "Multi-head Latent Attention: the KV cache, compressed", sections
// "The code" (the latent is x @ W_dkv and is the only thing cached) and
// "RoPE, and why the explanations stop here" (the decoupled key block is
// computed the ordinary way, rotated, and cached once for all heads);
// "DeepSeek V3 Multi-Head Latent Attention (MLA): How It Slashes KV Cache
// Memory", section "Low-Rank Key-Value Joint Compression".
//
// Three kernels share one epilogue:
//  * append_staged_kernel for decode-sized T (up to 256 tokens). The weight
//    read (d_model x R) dominates. Each CTA owns 4 packed columns. One thread
//    bulk-copies their d_model weights and the first 16 tokens' hidden states
//    into shared memory at entry, so the whole slice is in flight at once,
//    and later 16-token chunks reuse the staged weights.
//  * append_gemv_kernel, the same product with direct global loads, for
//    inputs the bulk copy cannot take (misaligned or very wide rows).
//  * append_gemm_kernel for bulk fills: a 64 x 64 register-tiled fp32 GEMM.
// The packed weight stores rotary dims i and i + d_r/2 in adjacent columns,
// so one thread (gemm) or one CTA (gemv) always holds both halves of a pair.
#include "device_common.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

struct AppendArgs {
  const double* inv_freq;
  const int32_t* seq_idx;
  const int32_t* pos;
  const int32_t* page_table;
  int B, max_blocks, num_blocks, T;
  uint32_t* err;
};

// Physical row of token t, or -1 (and an error bit) if its indices are bad.
__device__ __forceinline__ long long append_row(const AppendArgs& a, const Shape& s, int t) {
  const int b = a.seq_idx[t], p = a.pos[t];
  if (b < 0 || b >= a.B || p < 0 || p / s.bs >= a.max_blocks) {
    set_error(a.err, MLA_DEVERR_APPEND_INDEX);
    return -1;
  }
  const int page = a.page_table[static_cast<size_t>(b) * a.max_blocks + p / s.bs];
  if (page < 0 || page >= a.num_blocks) {
    set_error(a.err, MLA_DEVERR_PAGE_RANGE);
    return -1;
  }
  return static_cast<long long>(page) * s.bs + p % s.bs;
}

// Value of packed column pc after RoPE, given the pre-rotation values of the
// pair it belongs to (v_even: rotary dim i, v_odd: rotary dim i + d_r/2).
// Returns the cache column it lands in.
__device__ __forceinline__ int finish_column(const Shape& s, const double* inv_freq, int pc,
                                             float v_self, float v_even, float v_odd, int pos,
                                             float* out) {
  if (pc < s.d_c) {
    *out = v_self;
    return pc;
  }
  const int j = pc - s.d_c, i = j >> 1, e = j & 1, half = s.d_r / 2;
  float c, sn;
  rope_cos_sin(pos, inv_freq[i], &c, &sn);
  *out = e == 0 ? v_even * c - v_odd * sn : v_even * sn + v_odd * c;
  return s.d_c + i + e * half;
}

constexpr int GEMV_COLS = 4, GEMV_TOK = 8, GEMV_THREADS = 256;

// Requires d_model % Vec<T>::N == 0 and 16-byte aligned rows.
template <typename T>
__global__ void __launch_bounds__(GEMV_THREADS)
append_gemv_kernel(Shape s, const T* __restrict__ x, const T* __restrict__ Wp,
                   T* __restrict__ cache, AppendArgs a) {
  constexpr int V = Vec<T>::N;
  __shared__ float red[GEMV_THREADS / 32][GEMV_COLS * GEMV_TOK];
  __shared__ float res[GEMV_COLS * GEMV_TOK];
  const int R = s.R();
  const int col0 = blockIdx.x * GEMV_COLS;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int t0 = 0; t0 < a.T; t0 += GEMV_TOK) {
    float acc[GEMV_COLS][GEMV_TOK];
#pragma unroll
    for (int c = 0; c < GEMV_COLS; ++c)
#pragma unroll
      for (int t = 0; t < GEMV_TOK; ++t) acc[c][t] = 0.f;
    for (int k = threadIdx.x * V; k < s.d_model; k += GEMV_THREADS * V) {
      float wv[GEMV_COLS][V];
#pragma unroll
      for (int c = 0; c < GEMV_COLS; ++c) {
        if (col0 + c < R) {
          load_vec<T>(Wp + static_cast<size_t>(col0 + c) * s.d_model + k, wv[c]);
        } else {
#pragma unroll
          for (int i = 0; i < V; ++i) wv[c][i] = 0.f;
        }
      }
#pragma unroll
      for (int t = 0; t < GEMV_TOK; ++t) {
        if (t0 + t < a.T) {
          float xv[V];
          load_vec<T>(x + static_cast<size_t>(t0 + t) * s.d_model + k, xv);
#pragma unroll
          for (int c = 0; c < GEMV_COLS; ++c)
#pragma unroll
            for (int i = 0; i < V; ++i) acc[c][t] = fmaf(wv[c][i], xv[i], acc[c][t]);
        }
      }
    }
#pragma unroll
    for (int c = 0; c < GEMV_COLS; ++c)
#pragma unroll
      for (int t = 0; t < GEMV_TOK; ++t) {
        float v = acc[c][t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[warp][c * GEMV_TOK + t] = v;
      }
    __syncthreads();
    if (threadIdx.x < GEMV_COLS * GEMV_TOK) {
      float v = 0.f;
      for (int w = 0; w < GEMV_THREADS / 32; ++w) v += red[w][threadIdx.x];
      res[threadIdx.x] = v;
    }
    __syncthreads();
    if (threadIdx.x < GEMV_COLS * GEMV_TOK) {
      const int c = threadIdx.x / GEMV_TOK, t = threadIdx.x % GEMV_TOK;
      const int pc = col0 + c, tok = t0 + t;
      if (pc < R && tok < a.T) {
        const long long row = append_row(a, s, tok);
        if (row >= 0) {
          const int ce = c & ~1;  // even member of the pair inside this CTA
          float out;
          const int dst = finish_column(s, a.inv_freq, pc, res[c * GEMV_TOK + t],
                                        res[ce * GEMV_TOK + t], res[(ce + 1) * GEMV_TOK + t],
                                        a.pos[tok], &out);
          cache[row * R + dst] = from_f32<T>(out);
        }
      }
    }
    __syncthreads();
  }
}

constexpr int ST_COLS = 4, ST_TOK = 16, ST_THREADS = 256;
constexpr long long ST_WAIT = 2000000000LL;

// Dynamic shared memory: W slice [ST_COLS][d_model], then x chunk
// [ST_TOK][d_model], both in the input dtype; the barrier sits in static
// shared memory. Requires d_model * sizeof(T) % 16 == 0 and 16-byte aligned x.
template <typename T>
__global__ void __launch_bounds__(ST_THREADS)
append_staged_kernel(Shape s, const T* __restrict__ x, const T* __restrict__ Wp,
                     T* __restrict__ cache, AppendArgs a) {
  using namespace mla_ptx;
  constexpr int V = Vec<T>::N;
  extern __shared__ __align__(128) uint8_t st_raw[];
  T* ws = reinterpret_cast<T*>(st_raw);
  T* xs = ws + static_cast<size_t>(ST_COLS) * s.d_model;
  __shared__ uint64_t bar;
  __shared__ float red[ST_THREADS / 32][ST_COLS * 4];
  __shared__ float res[ST_COLS * ST_TOK];
  __shared__ int failed;
  const int R = s.R();
  const int col0 = blockIdx.x * ST_COLS;
  const int ncol = min(ST_COLS, R - col0);
  const uint32_t row_bytes = static_cast<uint32_t>(s.d_model) * sizeof(T);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int tg = threadIdx.x / 64, ks = threadIdx.x % 64;  // token group, k slice
  if (threadIdx.x == 0) {
    failed = 0;
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  int chunk = 0;
  for (int t0 = 0; t0 < a.T; t0 += ST_TOK, ++chunk) {
    const int nt = min(ST_TOK, a.T - t0);
    if (threadIdx.x == 0) {
      const uint32_t wbytes = chunk == 0 ? ncol * row_bytes : 0u;
      mbar_arrive_expect_tx(&bar, wbytes + nt * row_bytes);
      if (chunk == 0) bulk_load(ws, Wp + static_cast<size_t>(col0) * s.d_model, wbytes, &bar);
      bulk_load(xs, x + static_cast<size_t>(t0) * s.d_model, nt * row_bytes, &bar);
    }
    if (!mbar_wait(&bar, chunk & 1, ST_WAIT)) failed = 1;
    __syncthreads();
    if (failed) {
      if (threadIdx.x == 0) set_error(a.err, MLA_DEVERR_TIMEOUT);
      return;
    }
    float acc[ST_COLS][4];
#pragma unroll
    for (int c = 0; c < ST_COLS; ++c)
#pragma unroll
      for (int t = 0; t < 4; ++t) acc[c][t] = 0.f;
    for (int k = V * ks; k < s.d_model; k += 64 * V) {
      float wv[ST_COLS][V];
#pragma unroll
      for (int c = 0; c < ST_COLS; ++c) {
        if (c < ncol) {
          load_vec<T>(ws + static_cast<size_t>(c) * s.d_model + k, wv[c]);
        } else {
#pragma unroll
          for (int i = 0; i < V; ++i) wv[c][i] = 0.f;
        }
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int tt = 4 * tg + t;
        if (tt < nt) {
          float xv[V];
          load_vec<T>(xs + static_cast<size_t>(tt) * s.d_model + k, xv);
#pragma unroll
          for (int c = 0; c < ST_COLS; ++c)
#pragma unroll
            for (int i = 0; i < V; ++i) acc[c][t] = fmaf(wv[c][i], xv[i], acc[c][t]);
        }
      }
    }
#pragma unroll
    for (int c = 0; c < ST_COLS; ++c)
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float v = acc[c][t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[warp][c * 4 + t] = v;
      }
    __syncthreads();
    if (threadIdx.x < ST_COLS * ST_TOK) {
      const int c = threadIdx.x / ST_TOK, tt = threadIdx.x % ST_TOK;
      const int g = tt / 4, t = tt % 4;  // warps 2g and 2g+1 hold token group g
      res[threadIdx.x] = red[2 * g][c * 4 + t] + red[2 * g + 1][c * 4 + t];
    }
    __syncthreads();
    if (threadIdx.x < ST_COLS * ST_TOK) {
      const int c = threadIdx.x / ST_TOK, tt = threadIdx.x % ST_TOK;
      const int pc = col0 + c, tok = t0 + tt;
      if (c < ncol && tt < nt) {
        const long long row = append_row(a, s, tok);
        if (row >= 0) {
          const int ce = c & ~1;  // even member of the rotary pair inside this CTA
          float out;
          const int dst = finish_column(s, a.inv_freq, pc, res[c * ST_TOK + tt],
                                        res[ce * ST_TOK + tt], res[(ce + 1) * ST_TOK + tt],
                                        a.pos[tok], &out);
          cache[row * R + dst] = from_f32<T>(out);
        }
      }
    }
    __syncthreads();  // x chunk and res are reused
  }
}

constexpr int GM_BT = 64, GM_BC = 64, GM_BK = 32;

template <typename T>
__global__ void __launch_bounds__(256)
append_gemm_kernel(Shape s, const T* __restrict__ x, const T* __restrict__ Wp,
                   T* __restrict__ cache, AppendArgs a) {
  __shared__ float xs[GM_BK][GM_BT + 4];
  __shared__ float ws[GM_BK][GM_BC + 4];
  const int R = s.R();
  const int tok0 = blockIdx.x * GM_BT, col0 = blockIdx.y * GM_BC;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  // loader mapping: 64 rows x 32 k, 8 consecutive k per thread
  const int lr = threadIdx.x / 4, lk = (threadIdx.x % 4) * 8;
  for (int k0 = 0; k0 < s.d_model; k0 += GM_BK) {
    {
      const int t = tok0 + lr;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = k0 + lk + i;
        xs[lk + i][lr] =
            (t < a.T && k < s.d_model) ? to_f32<T>(x[static_cast<size_t>(t) * s.d_model + k]) : 0.f;
      }
      const int c = col0 + lr;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = k0 + lk + i;
        ws[lk + i][lr] =
            (c < R && k < s.d_model) ? to_f32<T>(Wp[static_cast<size_t>(c) * s.d_model + k]) : 0.f;
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < GM_BK; ++kk) {
      float xv[4], wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) wv[j] = ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int tok = tok0 + ty * 4 + i;
    if (tok >= a.T) continue;
    const long long row = append_row(a, s, tok);
    if (row < 0) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int pc = col0 + tx * 4 + j;
      if (pc >= R) continue;
      const int je = j & ~1;
      float out;
      const int dst =
          finish_column(s, a.inv_freq, pc, acc[i][j], acc[i][je], acc[i][je + 1], a.pos[tok], &out);
      cache[row * R + dst] = from_f32<T>(out);
    }
  }
}

template <typename T>
cudaError_t append_t(const Shape& s, const Weights* w, const void* x, AppendArgs a, void* cache,
                     cudaStream_t st) {
  const int R = s.R();
  const bool aligned = reinterpret_cast<uintptr_t>(x) % 16 == 0;
  const size_t staged_smem = sizeof(T) * static_cast<size_t>(ST_COLS + ST_TOK) * s.d_model;
  if (a.T <= 256 && aligned && s.d_model % Vec<T>::N == 0 && staged_smem <= 200 * 1024) {
    static int attr_bytes[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (staged_smem > 48 * 1024 &&
        (dev < 0 || dev >= 64 || attr_bytes[dev] < static_cast<int>(staged_smem))) {
      cudaError_t e = cudaFuncSetAttribute(append_staged_kernel<T>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(staged_smem));
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) attr_bytes[dev] = static_cast<int>(staged_smem);
    }
    const int grid = (R + ST_COLS - 1) / ST_COLS;
    append_staged_kernel<T><<<grid, ST_THREADS, staged_smem, st>>>(
        s, static_cast<const T*>(x), static_cast<const T*>(w->w_dkvr), static_cast<T*>(cache), a);
  } else if (a.T <= 32 && aligned && s.d_model % Vec<T>::N == 0) {
    const int grid = (R + GEMV_COLS - 1) / GEMV_COLS;
    append_gemv_kernel<T><<<grid, GEMV_THREADS, 0, st>>>(
        s, static_cast<const T*>(x), static_cast<const T*>(w->w_dkvr), static_cast<T*>(cache), a);
  } else {
    dim3 grid((a.T + GM_BT - 1) / GM_BT, (R + GM_BC - 1) / GM_BC);
    append_gemm_kernel<T><<<grid, 256, 0, st>>>(
        s, static_cast<const T*>(x), static_cast<const T*>(w->w_dkvr), static_cast<T*>(cache), a);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const Shape& s, mla_dtype dt, const Weights* w, const void* x,
                          const int32_t* seq_idx, const int32_t* pos, const int32_t* page_table,
                          int B, int max_blocks, void* cache, int num_blocks, int T,
                          uint32_t* err, cudaStream_t st) {
  AppendArgs a{w->inv_freq, seq_idx, pos, page_table, B, max_blocks, num_blocks, T, err};
  if (dt == MLA_F32) return append_t<float>(s, w, x, a, cache, st);
  return append_t<__nv_bfloat16>(s, w, x, a, cache, st);
}

}  // namespace mla
