// Full-fold variant of the decode layer: the hidden state x_q goes in and the
// layer output y comes out, with both up-projections folded into the
// neighbouring projections once, at load:
//
//   W_abs[h] = W_q,nope[h] W_uk[h]^T     (d_model x d_c)  query side
//   W_vo[h]  = W_uv[h] W_o[h]            (d_c x d_model)  output side
//
//   q_lat[t, h] = x_q[t] W_abs[h],   q_pe[t, h] = RoPE(x_q[t] W_qr[h], pos_t)
//   o_lat[t, h] = latent attention over the cache (the same kernels as the
//                 per-head path)
//   y[t]        = sum_h o_lat[t, h] W_vo[h]
//
// Sources: "Multi-head Latent Attention: the KV cache, compressed", sections
// "Store the archive, not the files" (W_abs = W_q W_uk^T, built once at
// load) and "The code" (absorb_q_into_latent; decoupled_score keeps the
// rotary block W_qr apart and rotates x_q W_qr at the query position);
// "Multi-head Latent Attention and KV Cache Compression", section "The
// absorption trick and decoupled RoPE" (the value up-projection folds into
// the output projection the same way).
//
// The first page warns that at DeepSeek's ratios the fold costs more than
// it saves ("Absorption: the part that makes it free"): W_abs is d_model x d_c
// per head where W_q,nope is d_model x d_nope, so the folded weights stream
// R/d_nope = 4.5x (query side) and d_model/d_v = 40x (output side) more bytes
// per step at DeepSeek-V2 shapes. It pays at small model widths.
//
// Folded weights are kept in fp32 (the product of two rounded matrices is
// not a value of the input dtype); the fold accumulates in fp64. The two
// x W products are HBM-bound weight streams: a CTA owns 1024 output columns
// (4 per thread) and 16 query rows, W arrives by TMA, and K is split across
// CTAs until the grid covers the SMs twice. The split partials are summed in
// a fixed order by a second kernel, so results are deterministic.
#include "device_common.cuh"
#include "plan.cuh"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace mla_ptx;

constexpr int XW_THREADS = 256;
constexpr int XW_VEC = 4;                      // output columns per thread
constexpr int XW_COLS = XW_THREADS * XW_VEC;   // output columns per CTA
constexpr int XW_ROWS = 16;                    // rows of A (query tokens) per CTA
constexpr int XW_KC = 64;                      // K chunk staged in shared memory
constexpr int QF_THREADS = 256;
constexpr int FOLD_THREADS = 256;

// TMA-ring form of the x W product (W rows 16-byte aligned). W arrives in
// 2-D tensor-map boxes of XR_BOXC columns x RS rows: four boxes cover a
// CTA's 1024 columns, and a stage is 32 KB whatever W's type (8 rows of
// fp32, 16 of bf16), so each request moves 8 KB. (One 1-D bulk copy per row,
// 2-4 KB each, left the copy engine request-bound.)
constexpr int XR_CONSUMERS = 256;               // 8 warps, 4 columns per thread
constexpr int XR_THREADS = XR_CONSUMERS + 32;   // + one producer warp
constexpr int XR_COLS = 4 * XR_CONSUMERS;       // output columns per CTA
constexpr int XR_BOXC = 256;                    // columns per tensor-map box
constexpr int XR_NBOX = XR_COLS / XR_BOXC;      // boxes per stage
constexpr int XR_NST = 3;                       // ring stages
constexpr int XR_KGRAN = 16;                    // K splits are multiples of every RS
constexpr int XR_KA = 192;                      // rows of A^T staged at a time
constexpr long long XR_WAIT = 2000000000LL;     // about 1 s at 2 GHz

template <typename TW>
struct XrRing {
  static constexpr int RS = 32 / static_cast<int>(sizeof(TW));  // W rows per stage
  static_assert(XR_KA % RS == 0, "a stage never straddles two A chunks");
  static_assert(XR_KGRAN % RS == 0, "splits hold whole stages");
};

template <typename TW>
struct XrSmem {
  TW w[XR_NST][XR_NBOX][XrRing<TW>::RS][XR_BOXC];  // ring of W boxes (32 KB per stage)
  float a[XR_KA][XW_ROWS];                          // A^T chunk, row index fastest
  uint64_t full[XR_NST], empty[XR_NST];
};

// Four consecutive W elements of a row, widened to fp32.
__device__ __forceinline__ float4 load_w4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float4 load_w4(const __nv_bfloat16* p) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                     __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
}

// out[z][m][n] = sum over k in split z of A[m][k] W[k][n], fp32 accumulation
// in k order. W is row-major [K][N] in TW; A is [M][K] in TA.
template <typename TA, typename TW>
__global__ void __launch_bounds__(XW_THREADS)
xw_kernel(const TA* __restrict__ A, int M, int K, const TW* __restrict__ W, int N,
          int k_split, float* __restrict__ out) {
  griddep_wait();  // A comes from the previous kernel (a no-op without programmatic launch)
  __shared__ __align__(16) float a_s[XW_KC][XW_ROWS];  // row index fastest
  const int n0 = blockIdx.x * XW_COLS + threadIdx.x * XW_VEC;
  const int m0 = blockIdx.y * XW_ROWS, mt = min(XW_ROWS, M - m0);
  const int kb = blockIdx.z * k_split, ke = min(K, kb + k_split);
  // one load of 4 consecutive W elements: rows must start at multiples of 4
  // elements (N % 4 == 0) from a base aligned to 4 elements
  const bool vec = (N % XW_VEC == 0) && n0 + XW_VEC <= N &&
                   reinterpret_cast<uintptr_t>(W) % (XW_VEC * sizeof(TW)) == 0;
  float acc[XW_ROWS][XW_VEC];
#pragma unroll
  for (int t = 0; t < XW_ROWS; ++t)
#pragma unroll
    for (int j = 0; j < XW_VEC; ++j) acc[t][j] = 0.f;

  for (int k0 = kb; k0 < ke; k0 += XW_KC) {
    const int kc = min(XW_KC, ke - k0);
    __syncthreads();  // the previous chunk is consumed
    for (int i = threadIdx.x; i < XW_KC * XW_ROWS; i += XW_THREADS) {
      const int t = i / XW_KC, k = i % XW_KC;  // consecutive threads walk k: coalesced in A
      a_s[k][t] = (t < mt && k < kc) ? to_f32<TA>(A[static_cast<size_t>(m0 + t) * K + k0 + k])
                                     : 0.f;
    }
    __syncthreads();
    if (n0 < N) {
#pragma unroll 4
      for (int k = 0; k < kc; ++k) {
        const TW* wp = W + static_cast<size_t>(k0 + k) * N + n0;
        float w[XW_VEC];
        if (vec) {
          const float4 v = load_w4(wp);
          w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
        } else {
#pragma unroll
          for (int j = 0; j < XW_VEC; ++j) w[j] = n0 + j < N ? to_f32<TW>(wp[j]) : 0.f;
        }
        const float4* av = reinterpret_cast<const float4*>(a_s[k]);
#pragma unroll
        for (int u = 0; u < XW_ROWS / 4; ++u) {
          const float4 a = av[u];
#pragma unroll
          for (int j = 0; j < XW_VEC; ++j) {
            acc[4 * u + 0][j] = fmaf(a.x, w[j], acc[4 * u + 0][j]);
            acc[4 * u + 1][j] = fmaf(a.y, w[j], acc[4 * u + 1][j]);
            acc[4 * u + 2][j] = fmaf(a.z, w[j], acc[4 * u + 2][j]);
            acc[4 * u + 3][j] = fmaf(a.w, w[j], acc[4 * u + 3][j]);
          }
        }
      }
    }
  }
  if (n0 >= N) return;
  float* o = out + static_cast<size_t>(blockIdx.z) * M * N;
  // rows start at multiples of 4 floats when N % 4 == 0: 16-byte stores need
  // only an aligned base (the caller's y may be any float pointer)
  const bool vec_out = vec && (reinterpret_cast<uintptr_t>(out) % 16 == 0);
#pragma unroll
  for (int t = 0; t < XW_ROWS; ++t) {
    if (t >= mt) break;
    float* orow = o + static_cast<size_t>(m0 + t) * N + n0;
    if (vec_out) {
      *reinterpret_cast<float4*>(orow) = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
    } else {
#pragma unroll
      for (int j = 0; j < XW_VEC; ++j)
        if (n0 + j < N) orow[j] = acc[t][j];
    }
  }
}

__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"r"(XR_CONSUMERS) : "memory");
}

// The same product as xw_kernel, with W streamed by TMA. One producer thread
// loads, per stage, four boxes (RS rows x 256 columns) of the CTA's columns
// into a 3-stage shared-memory ring; two CTAs per SM keep up to 192 KB of W
// in flight per SM without holding it in registers. The 256 consumer
// threads read their 4 elements of each row from shared memory and the 16 A
// values as four broadcast reads, and accumulate pairs of rows with
// the packed fp32x2 FMA (one IEEE fma per lane, so the sums are those of
// fmaf in the same order). Every wait is bounded: a timeout sets
// MLA_DEVERR_TIMEOUT, the consumers stop waiting, and the producer waits
// (bounded) for the copies it issued before the CTA exits.
template <typename TA, typename TW>
__global__ void __launch_bounds__(XR_THREADS, 2)
xw_ring_kernel(const __grid_constant__ CUtensorMap tmap_w, const TA* __restrict__ A, int M,
               int K, int N, int k_split, float* __restrict__ out, uint32_t* err) {
  constexpr int XR_RS = XrRing<TW>::RS;
  extern __shared__ uint8_t xr_raw[];
  XrSmem<TW>& sm = *reinterpret_cast<XrSmem<TW>*>(
      (reinterpret_cast<uintptr_t>(xr_raw) + 127) & ~static_cast<uintptr_t>(127));
  const int c0 = blockIdx.x * XR_COLS;
  const int m0 = blockIdx.y * XW_ROWS, mt = min(XW_ROWS, M - m0);
  const int kb = blockIdx.z * k_split, ke = min(K, kb + k_split);
  const int n_it = ke > kb ? (ke - kb + XR_RS - 1) / XR_RS : 0;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int st = 0; st < XR_NST; ++st) {
      mbar_init(&sm.full[st], 1);
      mbar_init(&sm.empty[st], XR_CONSUMERS / 32);
    }
    fence_mbarrier_init();
  }
  __syncthreads();

  if (warp == XR_CONSUMERS / 32) {  // producer
    if (lane != 0) return;
    // W is constant: the producer streams it without waiting for the
    // previous kernel (programmatic launch lets this overlap that kernel).
    // Boxes past N are not loaded; a box's columns past N and rows past K
    // arrive as zeros and still count their bytes.
    prefetch_tmap(&tmap_w);
    const int nbox = min(XR_NBOX, (N - c0 + XR_BOXC - 1) / XR_BOXC);
    const uint32_t stage_bytes = static_cast<uint32_t>(nbox * XR_RS * XR_BOXC * sizeof(TW));
    int it = 0;
    for (; it < n_it; ++it) {
      const int st = it % XR_NST;
      if (it >= XR_NST && !mbar_wait(&sm.empty[st], ((it / XR_NST) - 1) & 1, XR_WAIT)) {
        set_error(err, MLA_DEVERR_TIMEOUT);
        break;
      }
      const int k = kb + it * XR_RS;
      mbar_arrive_expect_tx(&sm.full[st], stage_bytes);
      for (int j = 0; j < nbox; ++j)
        tma_load_2d(sm.w[st][j], &tmap_w, c0 + j * XR_BOXC, k, &sm.full[st]);
    }
    // the copies issued last land before this thread (and so the CTA) exits
    for (int j = it > XR_NST ? it - XR_NST : 0; j < it; ++j)
      mbar_wait(&sm.full[j % XR_NST], (j / XR_NST) & 1, XR_WAIT);
    return;
  }

  griddep_wait();  // A comes from the previous kernel (a no-op without programmatic launch)
  const int tid = threadIdx.x;
  const int n0 = c0 + 4 * tid;
  const bool live = n0 < N;  // N % 4 == 0: all four columns are in range
  float2 acc[XW_ROWS / 2][4];  // acc[p][j]: rows 2p and 2p+1 of column n0 + j
#pragma unroll
  for (int p = 0; p < XW_ROWS / 2; ++p)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[p][j] = make_float2(0.f, 0.f);
  bool ok = true;
  int a_base = kb - XR_KA;
  for (int it = 0; it < n_it; ++it) {
    const int k = kb + it * XR_RS;
    if (k >= a_base + XR_KA) {  // the same decision in every consumer
      a_base = k;
      consumer_bar();  // the previous chunk is consumed
      const int ka = min(XR_KA, ke - k);
      for (int i = tid; i < XR_KA * XW_ROWS; i += XR_CONSUMERS) {
        const int t = i / XR_KA, kk = i % XR_KA;
        sm.a[kk][t] = (t < mt && kk < ka)
                          ? to_f32<TA>(A[static_cast<size_t>(m0 + t) * K + k + kk])
                          : 0.f;
      }
      consumer_bar();
    }
    const int st = it % XR_NST;
    if (ok) ok = mbar_wait(&sm.full[st], (it / XR_NST) & 1, XR_WAIT);
    const int rows = min(XR_RS, ke - k);
    if (live) {
#pragma unroll
      for (int r = 0; r < XR_RS; ++r) {
        if (r < rows) {
          const float4 w = load_w4(&sm.w[st][tid / 64][r][4 * (tid % 64)]);
          const float2 w0 = make_float2(w.x, w.x), w1 = make_float2(w.y, w.y);
          const float2 w2 = make_float2(w.z, w.z), w3 = make_float2(w.w, w.w);
          const float4* av = reinterpret_cast<const float4*>(sm.a[k - a_base + r]);
#pragma unroll
          for (int u = 0; u < XW_ROWS / 4; ++u) {
            const float4 a = av[u];
            const float2 lo = make_float2(a.x, a.y), hi = make_float2(a.z, a.w);
            acc[2 * u][0] = __ffma2_rn(lo, w0, acc[2 * u][0]);
            acc[2 * u][1] = __ffma2_rn(lo, w1, acc[2 * u][1]);
            acc[2 * u][2] = __ffma2_rn(lo, w2, acc[2 * u][2]);
            acc[2 * u][3] = __ffma2_rn(lo, w3, acc[2 * u][3]);
            acc[2 * u + 1][0] = __ffma2_rn(hi, w0, acc[2 * u + 1][0]);
            acc[2 * u + 1][1] = __ffma2_rn(hi, w1, acc[2 * u + 1][1]);
            acc[2 * u + 1][2] = __ffma2_rn(hi, w2, acc[2 * u + 1][2]);
            acc[2 * u + 1][3] = __ffma2_rn(hi, w3, acc[2 * u + 1][3]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[st]);
  }
  if (!ok && lane == 0) set_error(err, MLA_DEVERR_TIMEOUT);
  if (!live) return;
  float* o = out + static_cast<size_t>(blockIdx.z) * M * N;
  const bool vec_out = reinterpret_cast<uintptr_t>(out) % 16 == 0;
#pragma unroll
  for (int t = 0; t < XW_ROWS; ++t) {
    if (t >= mt) break;
    const int p = t / 2;
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = (t & 1) ? acc[p][j].y : acc[p][j].x;
    float* orow = o + static_cast<size_t>(m0 + t) * N + n0;
    if (vec_out) {
      *reinterpret_cast<float4*>(orow) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) orow[j] = v[j];
    }
  }
}

// out[i] = sum_z part[z][i], z in increasing order.
__global__ void __launch_bounds__(256)
sum_splits_kernel(const float* __restrict__ part, int S, size_t n, float* __restrict__ out) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float s = 0.f;
    for (int z = 0; z < S; ++z) s += part[static_cast<size_t>(z) * n + i];
    out[i] = s;
  }
}

// qabs[t, h] = out_scale * [q_lat | RoPE(q_rope, pos_t)] in T (fp32 for the
// CUDA-core attention, the cache dtype for the tensor-core one), from the fp32
// projection qpre[t][h*R + n]. One block per (token, QF_HEADS heads), so
// that each thread has only a few elements and the grid covers the SMs.
// Block 0 also writes the split-KV plan.
constexpr int QF_HEADS = 2;

template <typename T>
__global__ void __launch_bounds__(QF_THREADS)
q_finish_kernel(Shape s, const float* __restrict__ qpre, const uint64_t* __restrict__ rope_turns,
                const int32_t* __restrict__ seq_lens, int B, int n_q, int max_blocks, int TS,
                int G, int C, int K, float out_scale, T* __restrict__ qabs, int32_t* tiles,
                int32_t* prefix, long long* bounds, int32_t* first_b, uint32_t* err) {
  if (blockIdx.x == 0)
    write_plan<QF_THREADS>(seq_lens, B, n_q, max_blocks, s.bs, TS, G, C, K, tiles, prefix, bounds,
                           first_b, err);
  const int hg_n = (s.n_h + QF_HEADS - 1) / QF_HEADS;
  const int tok = blockIdx.x / hg_n, h0 = (blockIdx.x % hg_n) * QF_HEADS;
  const int nh = min(QF_HEADS, s.n_h - h0);
  const int b = tok / n_q, qi = tok % n_q;
  const int R = s.R(), half = s.d_r / 2, per_head = s.d_c + half;
  const int pos = seq_lens[b] - n_q + qi;
  const float* src = qpre + (static_cast<size_t>(tok) * s.n_h + h0) * R;
  T* dst = qabs + (static_cast<size_t>(tok) * s.n_h + h0) * R;
  for (int i = threadIdx.x; i < nh * per_head; i += QF_THREADS) {
    const int h = i / per_head, n = i % per_head;
    const float* sh = src + static_cast<size_t>(h) * R;
    T* dh = dst + static_cast<size_t>(h) * R;
    if (n < s.d_c) {
      dh[n] = from_f32<T>(sh[n] * out_scale);
    } else {
      const int k = n - s.d_c;
      const float x1 = sh[s.d_c + k], x2 = sh[s.d_c + k + half];
      float c, sn;
      rope_cos_sin(pos, rope_turns[k], &c, &sn);
      dh[s.d_c + k] = from_f32<T>((x1 * c - x2 * sn) * out_scale);
      dh[s.d_c + k + half] = from_f32<T>((x1 * sn + x2 * c) * out_scale);
    }
  }
}

// w_qf[m][h*R + n]: W_abs[h][m][n] = sum_k W_q[m][h*dq + k] W_uk[n][h*d_nope + k]
// for n < d_c, and the rotary query columns W_q[m][h*dq + d_nope + n - d_c]
// unchanged for n >= d_c.
template <typename T>
__global__ void __launch_bounds__(FOLD_THREADS)
fold_q_kernel(Shape s, const T* __restrict__ W_q, const T* __restrict__ W_uk,
              float* __restrict__ w_qf) {
  const int R = s.R(), dq = s.d_nope + s.d_r;
  const size_t NC = static_cast<size_t>(s.n_h) * R;
  const size_t total = static_cast<size_t>(s.d_model) * NC;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(idx / NC), col = static_cast<int>(idx % NC);
    const int h = col / R, n = col % R;
    const T* q = W_q + static_cast<size_t>(m) * s.n_h * dq + static_cast<size_t>(h) * dq;
    float v;
    if (n < s.d_c) {
      const T* u = W_uk + static_cast<size_t>(n) * s.n_h * s.d_nope + static_cast<size_t>(h) * s.d_nope;
      double acc = 0.0;
      for (int k = 0; k < s.d_nope; ++k)
        acc = fma(static_cast<double>(to_f32<T>(q[k])), static_cast<double>(to_f32<T>(u[k])), acc);
      v = static_cast<float>(acc);
    } else {
      v = to_f32<T>(q[s.d_nope + n - s.d_c]);
    }
    w_qf[idx] = v;
  }
}

// w_vo[h*d_c + c][m] = sum_k W_uv[c][h*d_v + k] W_o[h*d_v + k][m]
template <typename T>
__global__ void __launch_bounds__(FOLD_THREADS)
fold_o_kernel(Shape s, const T* __restrict__ W_uv, const T* __restrict__ W_o,
              float* __restrict__ w_vo) {
  const size_t total = static_cast<size_t>(s.n_h) * s.d_c * s.d_model;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(idx / s.d_model), m = static_cast<int>(idx % s.d_model);
    const int h = row / s.d_c, c = row % s.d_c;
    const T* u = W_uv + static_cast<size_t>(c) * s.n_h * s.d_v + static_cast<size_t>(h) * s.d_v;
    const T* o = W_o + static_cast<size_t>(h) * s.d_v * s.d_model + m;
    double acc = 0.0;
    for (int k = 0; k < s.d_v; ++k)
      acc = fma(static_cast<double>(to_f32<T>(u[k])),
                static_cast<double>(to_f32<T>(o[static_cast<size_t>(k) * s.d_model])), acc);
    w_vo[idx] = static_cast<float>(acc);
  }
}

int grid_for(size_t work, int sms) {
  const size_t blocks = (work + 255) / 256;
  return static_cast<int>(blocks < static_cast<size_t>(sms) * 16 ? (blocks ? blocks : 1)
                                                                 : static_cast<size_t>(sms) * 16);
}

template <typename T>
cudaError_t fold_t(const Shape& s, const void* W_q, const void* W_uk, const void* W_uv,
                   const void* W_o, FullWeights* w, int sms, cudaStream_t st) {
  const size_t nq = static_cast<size_t>(s.d_model) * s.n_h * s.R();
  const size_t no = static_cast<size_t>(s.n_h) * s.d_c * s.d_model;
  fold_q_kernel<T><<<grid_for(nq, sms), FOLD_THREADS, 0, st>>>(
      s, static_cast<const T*>(W_q), static_cast<const T*>(W_uk), w->w_qf);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fold_o_kernel<T><<<grid_for(no, sms), FOLD_THREADS, 0, st>>>(
      s, static_cast<const T*>(W_uv), static_cast<const T*>(W_o), w->w_vo);
  return cudaGetLastError();
}

template <typename T>
cudaError_t q_finish_t(const Shape& s, const uint64_t* rope_turns, const float* qpre,
                       const int32_t* seq_lens, int max_blocks, int B, int n_q, const Partition& p,
                       const WsView& ws, float out_scale, uint32_t* err, cudaStream_t st) {
  const long long blocks =
      static_cast<long long>(B) * n_q * ((s.n_h + QF_HEADS - 1) / QF_HEADS);
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  q_finish_kernel<T><<<static_cast<unsigned>(blocks), QF_THREADS, 0, st>>>(
      s, qpre, rope_turns, seq_lens, B, n_q, max_blocks, p.TS, p.G, p.C, p.K, out_scale,
      static_cast<T*>(ws.qabs), ws.tiles, ws.prefix, ws.bounds, ws.first_b, err);
  return cudaGetLastError();
}

// qabs = out_scale * q_abs, element by element, in T (the attention kernel's
// query type), from queries the caller has already absorbed and rotated
// (mla_decode_latent). Block 0 also writes the split-KV plan.
template <typename TI, typename T>
__global__ void __launch_bounds__(QF_THREADS)
latent_q_kernel(Shape s, const TI* __restrict__ q_abs, size_t n, const int32_t* __restrict__ seq_lens,
                int B, int n_q, int max_blocks, int TS, int G, int C, int K, float out_scale,
                T* __restrict__ qabs, int32_t* tiles, int32_t* prefix, long long* bounds,
                int32_t* first_b, uint32_t* err) {
  if (blockIdx.x == 0)
    write_plan<QF_THREADS>(seq_lens, B, n_q, max_blocks, s.bs, TS, G, C, K, tiles, prefix, bounds,
                           first_b, err);
  const size_t stride = static_cast<size_t>(gridDim.x) * QF_THREADS;
  const size_t first = static_cast<size_t>(blockIdx.x) * QF_THREADS + threadIdx.x;
  if constexpr (sizeof(TI) == 2 && sizeof(T) == 2) {
    // eight elements per 16-byte access where the caller's buffer allows it
    if (reinterpret_cast<uintptr_t>(q_abs) % 16 == 0 && n % 8 == 0) {
      for (size_t i = first; i < n / 8; i += stride) {
        uint4 v = reinterpret_cast<const uint4*>(q_abs)[i];
        TI* x = reinterpret_cast<TI*>(&v);
        uint4 o;
        T* y = reinterpret_cast<T*>(&o);
#pragma unroll
        for (int k = 0; k < 8; ++k) y[k] = from_f32<T>(to_f32<TI>(x[k]) * out_scale);
        reinterpret_cast<uint4*>(qabs)[i] = o;
      }
      return;
    }
  }
  for (size_t i = first; i < n; i += stride) qabs[i] = from_f32<T>(to_f32<TI>(q_abs[i]) * out_scale);
}

template <typename TI, typename T>
cudaError_t latent_q_t(const Shape& s, const void* q_abs, const int32_t* seq_lens, int max_blocks,
                       int B, int n_q, const Partition& p, const WsView& ws, float out_scale,
                       uint32_t* err, cudaStream_t st) {
  const size_t n = static_cast<size_t>(B) * n_q * s.n_h * s.R();
  const size_t blocks = (n / 8 + QF_THREADS) / QF_THREADS;
  latent_q_kernel<TI, T><<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), QF_THREADS, 0,
                           st>>>(s, static_cast<const TI*>(q_abs), n, seq_lens, B, n_q, max_blocks,
                                 p.TS, p.G, p.C, p.K, out_scale, static_cast<T*>(ws.qabs),
                                 ws.tiles, ws.prefix, ws.bounds, ws.first_b, err);
  return cudaGetLastError();
}

}  // namespace

// K is split so that the grid fills the two CTAs per SM that the ring kernel
// holds in one wave (tiles * S <= 2 * sms) without leaving most SMs idle:
// S = floor(2 sms / tiles), at least 1, in whole groups of XR_KGRAN rows.
XwPlan xw_plan(int M, int K, int N, int sms) {
  XwPlan p;
  const long long tiles = static_cast<long long>((N + XW_COLS - 1) / XW_COLS) *
                          ((M + XW_ROWS - 1) / XW_ROWS);
  const int stages = (K + XR_KGRAN - 1) / XR_KGRAN;
  long long S = tiles > 0 ? (2LL * sms) / tiles : 1;
  if (S > stages) S = stages;
  if (S < 1) S = 1;
  if (S > 65535) S = 65535;
  const int per = (stages + static_cast<int>(S) - 1) / static_cast<int>(S);
  p.k_split = per * XR_KGRAN;
  p.S = (K + p.k_split - 1) / p.k_split;
  if (p.S < 1) p.S = 1;
  return p;
}

size_t xw_part_floats(int M, int N, const XwPlan& p) {
  return p.S > 1 ? static_cast<size_t>(p.S) * M * N : 0;
}

// Launches one of the two forms, with programmatic dependent launch when
// pdl is set (the kernel's prologue and its W stream may then overlap the
// previous kernel; its reads of A wait for that kernel).
template <typename TA, typename TW>
cudaError_t xw_t(const void* A_, int M, int K, const void* W_, int N, int k_split, float* dst,
                 uint32_t* err, dim3 grid, bool pdl, cudaStream_t st) {
  const TA* A = static_cast<const TA*>(A_);
  const TW* W = static_cast<const TW*>(W_);
  // the tensor map needs a 16-byte aligned base and row stride
  bool ring = (static_cast<size_t>(N) * sizeof(TW)) % 16 == 0 &&
                    reinterpret_cast<uintptr_t>(W) % 16 == 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  CUtensorMap tm;
  if (ring) {
    TmapSpec spec = {};
    spec.dtype = sizeof(TW) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    spec.rank = 2;
    spec.base = W;
    spec.dims[0] = static_cast<uint64_t>(N);
    spec.dims[1] = static_cast<uint64_t>(K);
    spec.strides[0] = static_cast<uint64_t>(N) * sizeof(TW);
    spec.box[0] = XR_BOXC;
    spec.box[1] = XrRing<TW>::RS;
    spec.swizzle = CU_TENSOR_MAP_SWIZZLE_NONE;
    ring = get_tmap(spec, &tm);  // the register form takes what the encoder refuses
  }
  if (ring) {
    const int smem = static_cast<int>(sizeof(XrSmem<TW>)) + 128;
    cudaError_t e = cudaFuncSetAttribute(xw_ring_kernel<TA, TW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cfg.blockDim = dim3(XR_THREADS);
    cfg.dynamicSmemBytes = smem;
    return cudaLaunchKernelEx(&cfg, xw_ring_kernel<TA, TW>, tm, A, M, K, N, k_split, dst, err);
  }
  cfg.blockDim = dim3(XW_THREADS);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, xw_kernel<TA, TW>, A, M, K, W, N, k_split, dst);
}

cudaError_t launch_xw(mla_dtype a_dt, const void* A, int M, int K, mla_dtype w_dt,
                      const void* W, int N, float* out, float* part, const XwPlan& p,
                      uint32_t* err, bool pdl, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  if (M > 65535 * XW_ROWS) return cudaErrorInvalidValue;
  static_assert(XR_COLS == XW_COLS, "both forms tile the columns alike");
  dim3 grid((N + XW_COLS - 1) / XW_COLS, (M + XW_ROWS - 1) / XW_ROWS, p.S);
  float* dst = p.S > 1 ? part : out;
  using bf16 = __nv_bfloat16;
  cudaError_t e;
  if (a_dt == MLA_F32 && w_dt == MLA_F32)
    e = xw_t<float, float>(A, M, K, W, N, p.k_split, dst, err, grid, pdl, st);
  else if (a_dt == MLA_F32)
    e = xw_t<float, bf16>(A, M, K, W, N, p.k_split, dst, err, grid, pdl, st);
  else if (w_dt == MLA_F32)
    e = xw_t<bf16, float>(A, M, K, W, N, p.k_split, dst, err, grid, pdl, st);
  else
    e = xw_t<bf16, bf16>(A, M, K, W, N, p.k_split, dst, err, grid, pdl, st);
  if (e != cudaSuccess || p.S == 1) return e;
  return launch_sum_splits(part, p.S, static_cast<size_t>(M) * N, out, st);
}

cudaError_t launch_sum_splits(const float* part, int S, size_t n, float* out, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const size_t blocks = (n + 255) / 256;
  sum_splits_kernel<<<static_cast<int>(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(part, S, n,
                                                                                       out);
  return cudaGetLastError();
}

cudaError_t launch_fold_full(const Shape& s, mla_dtype dt, const void* W_q, const void* W_uk,
                             const void* W_uv, const void* W_o, FullWeights* w, int sms,
                             cudaStream_t st) {
  if (dt == MLA_F32) return fold_t<float>(s, W_q, W_uk, W_uv, W_o, w, sms, st);
  return fold_t<__nv_bfloat16>(s, W_q, W_uk, W_uv, W_o, w, sms, st);
}

cudaError_t launch_q_finish(const Shape& s, mla_dtype dt, const uint64_t* rope_turns,
                            const float* qpre, const int32_t* seq_lens, int max_blocks, int B,
                            int n_q, const Partition& p, const WsView& ws, float out_scale,
                            bool q_f32, uint32_t* err, cudaStream_t st) {
  if (dt == MLA_F32 || q_f32)
    return q_finish_t<float>(s, rope_turns, qpre, seq_lens, max_blocks, B, n_q, p, ws, out_scale,
                             err, st);
  return q_finish_t<__nv_bfloat16>(s, rope_turns, qpre, seq_lens, max_blocks, B, n_q, p, ws,
                                   out_scale, err, st);
}

cudaError_t launch_latent_q(const Shape& s, mla_dtype dt, const void* q_abs,
                            const int32_t* seq_lens, int max_blocks, int B, int n_q,
                            const Partition& p, const WsView& ws, float out_scale, bool q_f32,
                            uint32_t* err, cudaStream_t st) {
  if (dt == MLA_F32)
    return latent_q_t<float, float>(s, q_abs, seq_lens, max_blocks, B, n_q, p, ws, out_scale, err,
                                    st);
  if (q_f32)
    return latent_q_t<__nv_bfloat16, float>(s, q_abs, seq_lens, max_blocks, B, n_q, p, ws,
                                            out_scale, err, st);
  return latent_q_t<__nv_bfloat16, __nv_bfloat16>(s, q_abs, seq_lens, max_blocks, B, n_q, p, ws,
                                                  out_scale, err, st);
}

}  // namespace mla
