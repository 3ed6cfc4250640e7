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
// bf16 appends run on the tensor cores (append_tc_kernel below, a split-K
// tcgen05 GEMM of up to 256 tokens per launch; longer bulk fills are
// consecutive launches). The CUDA-core kernels take fp32 and the shapes the
// tensor-core kernel does not; three of them share one epilogue:
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
#include "tmap.h"

namespace mla {
namespace {

struct AppendArgs {
  const uint64_t* rope_turns;
  const int32_t* seq_idx;
  const int32_t* pos;
  const int32_t* page_table;
  int B, max_blocks, num_blocks, T;
  uint32_t* err;
  // When set, the rows go here instead, in fp32 and dense ([T][R], row t
  // for token t, no paging): the input of the fp8 row quantiser.
  float* rows_out;
};

// Physical row of token t, or -1 (and an error bit) if its indices are bad.
// In the dense fp32 mode every token has a row (the quantiser checks the
// indices when it places the rows).
__device__ __forceinline__ long long append_row(const AppendArgs& a, const Shape& s, int t) {
  if (a.rows_out) return t;
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

// Stores the finished value of cache column `dst` of the row returned by
// append_row: into the paged cache in T, or in fp32 into the dense rows.
template <typename T>
__device__ __forceinline__ void put_value(const AppendArgs& a, T* cache, long long row, int R,
                                          int dst, float v) {
  if (a.rows_out)
    a.rows_out[row * R + dst] = v;
  else
    cache[row * R + dst] = from_f32<T>(v);
}

// Value of packed column pc after RoPE, given the pre-rotation values of the
// pair it belongs to (v_even: rotary dim i, v_odd: rotary dim i + d_r/2).
// Returns the cache column it lands in.
__device__ __forceinline__ int finish_column(const Shape& s, const uint64_t* rope_turns, int pc,
                                             float v_self, float v_even, float v_odd, int pos,
                                             float* out) {
  if (pc < s.d_c) {
    *out = v_self;
    return pc;
  }
  const int j = pc - s.d_c, i = j >> 1, e = j & 1, half = s.d_r / 2;
  float c, sn;
  rope_cos_sin(pos, rope_turns[i], &c, &sn);
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
          const int dst = finish_column(s, a.rope_turns, pc, res[c * GEMV_TOK + t],
                                        res[ce * GEMV_TOK + t], res[(ce + 1) * GEMV_TOK + t],
                                        a.pos[tok], &out);
          put_value<T>(a, cache, row, R, dst, out);
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
          const int dst = finish_column(s, a.rope_turns, pc, res[c * ST_TOK + tt],
                                        res[ce * ST_TOK + tt], res[(ce + 1) * ST_TOK + tt],
                                        a.pos[tok], &out);
          put_value<T>(a, cache, row, R, dst, out);
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
          finish_column(s, a.rope_turns, pc, acc[i][j], acc[i][je], acc[i][je + 1], a.pos[tok], &out);
      put_value<T>(a, cache, row, R, dst, out);
    }
  }
}

// ---- tensor-core split-K path for decode-sized batches of bf16 tokens ----
//
// D[R x T] = Wp[R x d_model] x^T. The R packed columns are cut into blocks of
// 128 (MMA M; TMA zero-fills the rows past R) and d_model into KC slices (KC
// = 16, or 8 where clusters of 16 cannot be resident), one CTA each. The KC
// CTAs of a column block form one cluster: each stages its weight slice (the
// only large read) and the tokens' matching hidden-state slice with TMA,
// multiplies them into TMEM (N = tokens), and parks the fp32 partial in
// shared memory. After a cluster barrier CTA r sums rows [r 128/KC,
// (r + 1) 128/KC) over all KC partials through distributed shared memory
// (fixed order, so the result does not depend on timing), applies RoPE to the
// rotary pairs (adjacent rows of the packed weight) and writes the cache
// entries.
constexpr int AT_THREADS = 128;
constexpr int AT_MAX_TOK = 256;  // tokens per launch (the MMA N of one CTA)
constexpr uint32_t AT_WBOX = 128 * 128;  // 128 rows x 64 bf16
constexpr long long AT_WAIT = 2000000000LL;

__device__ __forceinline__ uint64_t at_desc(const uint8_t* p, uint32_t byte_off) {
  using namespace mla_ptx;
  return smem_desc(smem_u32(p) + byte_off, 16, 1024, kSwizzle128B);
}

__global__ void __launch_bounds__(AT_THREADS, 1)
append_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                 Shape s, int kcn, int nkb, int N, uint32_t tmem_cols,
                 __nv_bfloat16* __restrict__ cache, AppendArgs a) {
  using namespace mla_ptx;
  extern __shared__ uint8_t at_raw[];
  uint8_t* A = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(at_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  uint8_t* X = A + nkb * AT_WBOX;                             // nkb boxes of N rows x 128 B
  // [128 rows][N + 1] fp32 partial: the padded row keeps the 32 rows a warp
  // writes per column in 32 different banks
  float* red = reinterpret_cast<float*>(X + nkb * N * 128);
  const int NP = N + 1;
  __shared__ uint64_t full, done;
  __shared__ uint32_t tmem_base;
  const uint32_t kc = cluster_ctarank();
  const int mb = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int R = s.R();
  if (threadIdx.x == 0) {
    mbar_init(&full, 1);
    mbar_init(&done, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  // With programmatic dependent launch this CTA may start while the previous
  // kernel still runs. The packed weights are complete and never written
  // once their handle exists, so the weight slice is loaded at once; the
  // hidden states and the cache are touched only after the wait for that
  // kernel.
  const int k0 = static_cast<int>(kc) * nkb * 64;
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_x);
    mbar_arrive_expect_tx(&full, nkb * (AT_WBOX + N * 128));
    for (int j = 0; j < nkb; ++j) tma_load_2d(A + j * AT_WBOX, &tmap_w, k0 + 64 * j, mb * 128, &full);
  }
  griddep_wait();
  if (threadIdx.x == 0) {
    for (int j = 0; j < nkb; ++j) tma_load_2d(X + j * N * 128, &tmap_x, k0 + 64 * j, 0, &full);
    if (mbar_wait(&full, 0, AT_WAIT)) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, N, false, false);
      for (int j = 0; j < nkb; ++j)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16_ss(tmem, at_desc(A + j * AT_WBOX, 32 * k), at_desc(X + j * N * 128, 32 * k),
                      idesc, (j > 0 || k > 0) ? 1u : 0u);
    } else {
      set_error(a.err, MLA_DEVERR_TIMEOUT);
    }
    mma_commit(&done);  // arrives once the MMAs (if any) are done
  }
  // the next kernel (the query absorption) may be scheduled now; it waits
  // for this grid before it reads anything this kernel writes
  griddep_launch_dependents();
  // partial of this K slice: row (packed column) per lane, token per TMEM column
  const bool ok = mbar_wait(&done, 0, 2 * AT_WAIT);
  tc_fence_after();
  {
    const int row = 32 * warp + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    for (int c0 = 0; c0 < N; c0 += 16) {
      float v[16];
      tmem_ld16(tmem + lane_base + c0, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) red[row * NP + c0 + i] = ok ? v[i] : 0.f;
    }
  }
  if (!ok && threadIdx.x == 0) set_error(a.err, MLA_DEVERR_TIMEOUT);
  tc_fence_before();
  cluster_sync();  // every partial of the cluster is in place
  // CTA kc reduces its 128 / kcn rows: row pairs x N tokens
  const int rows = 128 / kcn;
  for (int it = threadIdx.x; it < (rows / 2) * N; it += AT_THREADS) {
    const int pr = it / N, t = it % N;
    const int r0 = rows * static_cast<int>(kc) + 2 * pr;  // even row of the pair
    const int pc0 = mb * 128 + r0;
    if (t >= a.T || pc0 >= R) continue;
    float p0[16], p1[16];
#pragma unroll
    for (int src = 0; src < 16; ++src) {
      if (src < kcn) {
        const float* r = map_to_rank(red, static_cast<uint32_t>(src));
        p0[src] = r[r0 * NP + t];
        p1[src] = r[(r0 + 1) * NP + t];
      } else {
        p0[src] = p1[src] = 0.f;
      }
    }
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int src = 0; src < 16; ++src) {
      v0 += p0[src];
      v1 += p1[src];
    }
    const long long row = append_row(a, s, t);
    if (row < 0) continue;
    float out;
    int dst = finish_column(s, a.rope_turns, pc0, v0, v0, v1, a.pos[t], &out);
    put_value<__nv_bfloat16>(a, cache, row, R, dst, out);
    if (pc0 + 1 < R) {
      dst = finish_column(s, a.rope_turns, pc0 + 1, v1, v0, v1, a.pos[t], &out);
      put_value<__nv_bfloat16>(a, cache, row, R, dst, out);
    }
  }
  cluster_sync();  // no CTA leaves while a peer may still read its partial
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// Dynamic shared memory of append_tc_kernel for N tokens and nkb boxes.
size_t append_tc_smem(int nkb, int N) {
  return 1024 + static_cast<size_t>(nkb) * (AT_WBOX + N * 128) + static_cast<size_t>(128) * (N + 1) * 4;
}

// Whether clusters of kcn CTAs of append_tc_kernel, each with `smem` bytes,
// can be resident.
bool append_tc_clusters_ok(int kcn, size_t smem) {
  // (the kernel's few static bytes count against the same 227 KB, so the
  // dynamic limit is raised to what this launch needs, not to the maximum)
  static size_t attr_bytes[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || attr_bytes[dev] < smem) {
    if (cudaFuncSetAttribute(append_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1) != cudaSuccess ||
        cudaFuncSetAttribute(append_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (dev >= 0 && dev < 64) attr_bytes[dev] = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kcn, 1, 1);
  cfg.blockDim = dim3(AT_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kcn;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const bool ok = cudaOccupancyMaxActiveClusters(&n, append_tc_kernel, &cfg) == cudaSuccess && n >= 1;
  cudaGetLastError();
  return ok;
}

// Cluster size chosen by launch_append_tc for these sizes, or 0 if the path
// does not apply (for diagnostics).
int append_tc_cluster_size(const Shape& s, int T, int* nkb_out, size_t* smem_out) {
  const int N = ((T + 15) / 16) * 16;
  if (T < 1 || N > AT_MAX_TOK || s.d_c % 2 != 0) return 0;
  for (int kcn : {16, 8}) {
    if (s.d_model % (kcn * 64) != 0) continue;
    const int nkb = s.d_model / (kcn * 64);
    const size_t smem = append_tc_smem(nkb, N);
    if (smem > 227 * 1024 - 1024 || !append_tc_clusters_ok(kcn, smem)) continue;
    *nkb_out = nkb;
    *smem_out = smem;
    return kcn;
  }
  return 0;
}

// Launches the split-K path if it applies; returns false (nothing launched)
// otherwise.
bool launch_append_tc(const Shape& s, const Weights* w, const void* x, const AppendArgs& a,
                      void* cache, cudaStream_t st, cudaError_t* err) {
  // (rotary pairs must sit in adjacent, even-aligned rows of a CTA's rows)
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0) return false;
  int nkb = 0;
  size_t smem = 0;
  const int kcn = append_tc_cluster_size(s, a.T, &nkb, &smem);
  if (kcn == 0) return false;
  const int N = ((a.T + 15) / 16) * 16;
  TmapSpec ws{};
  ws.dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  ws.rank = 2;
  ws.base = w->w_dkvr;
  ws.dims[0] = s.d_model;
  ws.dims[1] = s.R();
  ws.strides[0] = static_cast<uint64_t>(s.d_model) * 2;
  ws.box[0] = 64;
  ws.box[1] = 128;
  ws.swizzle = CU_TENSOR_MAP_SWIZZLE_128B;
  TmapSpec xs{};
  xs.dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  xs.rank = 2;
  xs.base = x;
  xs.dims[0] = s.d_model;
  xs.dims[1] = a.T;
  xs.strides[0] = static_cast<uint64_t>(s.d_model) * 2;
  xs.box[0] = 64;
  xs.box[1] = N;
  xs.swizzle = CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap tw, tx;
  if (!get_tmap(ws, &tw) || !get_tmap(xs, &tx)) return false;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(N)) cols *= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kcn, (s.R() + 127) / 128, 1);
  cfg.blockDim = dim3(AT_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kcn;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the previous kernel finishes (see the kernel's wait)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  *err = cudaLaunchKernelEx(&cfg, append_tc_kernel, tw, tx, s, kcn, nkb, N, cols,
                            static_cast<__nv_bfloat16*>(cache), a);
  return true;
}

// ---- tensor-core GEMM path for many bf16 tokens ----
//
// D[R x T] = Wp x^T in tiles of 128 packed columns x 128 tokens (MMA M and
// N), one CTA per tile, each over the whole of d_model: thread 0 streams the
// weight rows and the tokens' hidden states through a 6-stage TMA ring of
// 64-wide K chunks, thread 32 issues 4 MMAs per chunk into one TMEM
// accumulator, and no partial sum leaves the CTA. The four warps then read
// the accumulator (lane = packed column, so a rotary pair sits in two
// adjacent lanes), apply RoPE with the partner's value from a shuffle, and
// write each token's row. This is the path for bulk fills and prefill
// chunks, where the split-K kernel's whole-slice staging does not fit in
// shared memory.
constexpr int MM_N = 128;                // tokens per CTA
constexpr int MM_STAGES = 6;
constexpr uint32_t MM_ABOX = 128 * 128;  // 128 packed rows x 64 bf16
constexpr uint32_t MM_BBOX = MM_N * 128; // 128 tokens x 64 bf16

struct __align__(1024) MmSmem {
  uint8_t a[MM_STAGES][MM_ABOX];
  uint8_t b[MM_STAGES][MM_BBOX];
  uint64_t full[MM_STAGES], empty[MM_STAGES], done;
  long long row[MM_N];                   // cache row of each token of the tile (-1: skip)
  int pos[MM_N];
  uint32_t tmem_base;
};

__global__ void __launch_bounds__(128, 1)
append_mm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                 Shape s, int nk, __nv_bfloat16* __restrict__ cache, AppendArgs a) {
  using namespace mla_ptx;
  extern __shared__ uint8_t mm_raw[];
  MmSmem& sm = *reinterpret_cast<MmSmem*>((reinterpret_cast<uintptr_t>(mm_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  const int mb = blockIdx.x, t0 = blockIdx.y * MM_N;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int R = s.R();
  constexpr uint32_t STAGE_TX = MM_ABOX + MM_BBOX;
  if (threadIdx.x == 0) {
    for (int i = 0; i < MM_STAGES; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    mbar_init(&sm.done, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&sm.tmem_base, MM_N);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (threadIdx.x == 0) {
    // The packed weights are complete and never written once their handle
    // exists: their first chunks are requested before the wait for the
    // previous kernel; the hidden states only after it.
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_x);
    const int pre = min(nk, MM_STAGES);
    for (int i = 0; i < pre; ++i) {
      mbar_arrive_expect_tx(&sm.full[i], STAGE_TX);
      tma_load_2d(sm.a[i], &tmap_w, 64 * i, mb * 128, &sm.full[i]);
    }
    griddep_wait();
    for (int i = 0; i < pre; ++i) tma_load_2d(sm.b[i], &tmap_x, 64 * i, t0, &sm.full[i]);
    int issued = pre;
    bool ok = true;
    for (int i = MM_STAGES; i < nk; ++i) {
      const int st = i % MM_STAGES;
      if (!mbar_wait(&sm.empty[st], ((i / MM_STAGES) - 1) & 1, AT_WAIT)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(&sm.full[st], STAGE_TX);
      tma_load_2d(sm.a[st], &tmap_w, 64 * i, mb * 128, &sm.full[st]);
      tma_load_2d(sm.b[st], &tmap_x, 64 * i, t0, &sm.full[st]);
      issued = i + 1;
    }
    if (!ok) {
      set_error(a.err, MLA_DEVERR_TIMEOUT);
      // the loads already issued land before the CTA may exit
      for (int i = max(0, issued - MM_STAGES); i < issued; ++i)
        mbar_wait(&sm.full[i % MM_STAGES], (i / MM_STAGES) & 1, AT_WAIT);
    }
  } else if (threadIdx.x == 32) {
    const uint32_t idesc = idesc_bf16_f32(128, MM_N, false, false);
    bool ok = true;
    for (int i = 0; i < nk; ++i) {
      const int st = i % MM_STAGES;
      if (!mbar_wait(&sm.full[st], (i / MM_STAGES) & 1, AT_WAIT)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_bf16_ss(tmem, at_desc(sm.a[st], 32 * k), at_desc(sm.b[st], 32 * k), idesc,
                    (i > 0 || k > 0) ? 1u : 0u);
      mma_commit(&sm.empty[st]);
    }
    if (!ok) set_error(a.err, MLA_DEVERR_TIMEOUT);
    mma_commit(&sm.done);  // arrives once every MMA issued above is done
  }
  griddep_wait();  // (returns at once in the thread that already waited)
  // the next kernel may be scheduled now; it waits for this grid before it
  // reads anything this kernel writes
  griddep_launch_dependents();
  // the tile's tokens: cache row and position, once each
  {
    const int t = t0 + threadIdx.x;
    long long r = -1;
    int p = 0;
    if (t < a.T) {
      r = append_row(a, s, t);
      p = a.pos[t];
    }
    sm.row[threadIdx.x] = r;
    sm.pos[threadIdx.x] = p;
  }
  __syncthreads();
  const bool ok = mbar_wait(&sm.done, 0, 4 * AT_WAIT);
  tc_fence_after();
  if (!ok && threadIdx.x == 0) set_error(a.err, MLA_DEVERR_TIMEOUT);
  const int pc = mb * 128 + 32 * warp + lane;  // packed column of this lane
  const bool even = (lane & 1) == 0;
  const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
  for (int c0 = 0; c0 < MM_N && t0 + c0 < a.T; c0 += 16) {
    float v[16];
    tmem_ld16(tmem + lane_base + c0, v);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float partner = __shfl_xor_sync(0xffffffffu, v[i], 1);
      const long long row = sm.row[c0 + i];
      if (!ok || row < 0 || pc >= R) continue;
      float out;
      const int dst = finish_column(s, a.rope_turns, pc, v[i], even ? v[i] : partner,
                                    even ? partner : v[i], sm.pos[c0 + i], &out);
      put_value<__nv_bfloat16>(a, cache, row, R, dst, out);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, MM_N);
  }
}

// Launches the GEMM path if it applies (bf16, d_model a multiple of 64,
// 16-byte aligned x); returns false (nothing launched) otherwise.
bool launch_append_mm(const Shape& s, const Weights* w, const void* x, const AppendArgs& a,
                      void* cache, cudaStream_t st, cudaError_t* err) {
  if (reinterpret_cast<uintptr_t>(x) % 16 != 0 || s.d_model % 64 != 0 || s.R() % 2 != 0) return false;
  TmapSpec ws{};
  ws.dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  ws.rank = 2;
  ws.base = w->w_dkvr;
  ws.dims[0] = s.d_model;
  ws.dims[1] = s.R();
  ws.strides[0] = static_cast<uint64_t>(s.d_model) * 2;
  ws.box[0] = 64;
  ws.box[1] = 128;
  ws.swizzle = CU_TENSOR_MAP_SWIZZLE_128B;
  TmapSpec xs{};
  xs.dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  xs.rank = 2;
  xs.base = x;
  xs.dims[0] = s.d_model;
  xs.dims[1] = a.T;
  xs.strides[0] = static_cast<uint64_t>(s.d_model) * 2;
  xs.box[0] = 64;
  xs.box[1] = MM_N;
  xs.swizzle = CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap tw, tx;
  if (!get_tmap(ws, &tw) || !get_tmap(xs, &tx)) return false;
  const size_t smem = sizeof(MmSmem) + 1024;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    if (cudaFuncSetAttribute(append_mm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((s.R() + 127) / 128, (a.T + MM_N - 1) / MM_N, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  // may start while the previous kernel finishes (see the kernel's wait)
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  *err = cudaLaunchKernelEx(&cfg, append_mm_kernel, tw, tx, s, s.d_model / 64,
                            static_cast<__nv_bfloat16*>(cache), a);
  return true;
}

template <typename T>
cudaError_t append_t(const Shape& s, const Weights* w, const void* x, AppendArgs a, void* cache,
                     cudaStream_t st) {
  const int R = s.R();
  const bool aligned = reinterpret_cast<uintptr_t>(x) % 16 == 0;
  if constexpr (sizeof(T) == 2) {
    // decode-sized batches: the split-K kernel, whose whole weight slice is
    // in flight at once; larger ones (or where its staging does not fit):
    // the tile GEMM
    cudaError_t e = cudaSuccess;
    if (a.T <= AT_MAX_TOK && launch_append_tc(s, w, x, a, cache, st, &e)) return e;
    if (launch_append_mm(s, w, x, a, cache, st, &e)) return e;
  }
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
  AppendArgs a{w->rope_turns, seq_idx, pos, page_table, B, max_blocks, num_blocks, T, err,
               nullptr};
  if (dt == MLA_F32) return append_t<float>(s, w, x, a, cache, st);
  return append_t<__nv_bfloat16>(s, w, x, a, cache, st);
}

cudaError_t launch_append_rows_f32(const Shape& s, mla_dtype dt, const Weights* w, const void* x,
                                   const int32_t* seq_idx, const int32_t* pos, int T,
                                   float* rows, uint32_t* err, cudaStream_t st) {
  AppendArgs a{w->rope_turns, seq_idx, pos, nullptr, 1, 1, 1, T, err, rows};
  if (dt == MLA_F32) return append_t<float>(s, w, x, a, nullptr, st);
  return append_t<__nv_bfloat16>(s, w, x, a, nullptr, st);
}

}  // namespace mla
