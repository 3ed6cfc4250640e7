// a3 (CUDA-core variant): split-KV attention of absorbed queries over the
// paged latent cache, in fp32 FMA. Used for fp32 caches and for shapes the
// tensor-core kernel does not cover.
//
//   s_j   = (q_lat . c_j + q_pe . k_rope_j) * scale,   j <= pos_q
//   O_lat = sum_j softmax(s)_j c_j                      (online softmax)
//
// Sources: "Multi-head Latent Attention: the KV cache, compressed", sections
// "Absorption: the part that makes it free" (scores against the latent,
// keys never built) and "RoPE, and why the explanations stop here" (score =
// content part + decoupled RoPE part); "Multi-head Latent Attention and KV
// Cache Compression", section "The absorption trick and decoupled RoPE"
// (the value side is up-projected after the weighted sum).
//
// One CTA walks a contiguous range of (group, sequence, 64-token tile) work
// items. A group is 16 query rows. Each piece of the range writes a partial
// (O_lat / l, log-sum-exp) to its workspace slot. The combine kernel merges
// the partials.
#include <cmath>

#include "device_common.cuh"

namespace mla {
namespace {

constexpr int SG_ROWS = 16, SG_SUB = 16, SG_THREADS = 256, SG_MAXK = 32;  // d_c <= 512

template <typename T>
__global__ void __launch_bounds__(SG_THREADS)
attend_simt_kernel(Shape s, const T* __restrict__ cache, int num_blocks,
                   const int32_t* __restrict__ page_table, int max_blocks, int B, int n_q,
                   Partition p, const float* __restrict__ qabs, const int32_t* __restrict__ tiles,
                   const int32_t* __restrict__ prefix, const long long* __restrict__ bounds,
                   const int32_t* __restrict__ seq_lens, float* __restrict__ part_o,
                   float* __restrict__ part_lse, uint32_t* err) {
  extern __shared__ float sm[];
  const int R = s.R(), RP = R + 1;
  float* qs = sm;                      // [16][RP]
  float* ks = qs + SG_ROWS * RP;       // [16][RP]
  float* ps = ks + SG_SUB * RP;        // [16][16]
  float* alph = ps + SG_ROWS * SG_SUB; // [16]

  const int tid = threadIdx.x;
  const int r = tid / 16, c16 = tid % 16;  // score: row r, token c16; O: row r, dims c16 + 16k
  const int rows_total = n_q * s.n_h;
  const long long T_all = prefix[B];
  const long long N = T_all * p.G;
  if (N == 0) return;
  long long it = bounds[blockIdx.x];
  const long long end = bounds[blockIdx.x + 1];
  const float scale_log2 = s.scale * 1.4426950408889634f;

  while (it < end) {
    // locate (g, b, t) of item `it`
    const int g = static_cast<int>(it / T_all);
    const long long rem = it % T_all;
    int lo = 0, hi = B;  // largest b with prefix[b] <= rem
    while (hi - lo > 1) {
      const int mid = (lo + hi) / 2;
      if (prefix[mid] <= rem) lo = mid; else hi = mid;
    }
    const int b = lo;  // prefix[b] <= rem < prefix[b + 1], so tiles[b] > 0
    const int t_first = static_cast<int>(rem - prefix[b]);
    const long long piece_end = min(end, static_cast<long long>(g) * T_all + prefix[b] + tiles[b]);
    const int t_last = t_first + static_cast<int>(piece_end - it) - 1;
    const int L = seq_lens[b];

    // query rows of this group
    __syncthreads();
    for (int i = tid; i < SG_ROWS * R; i += SG_THREADS) {
      const int rr = i / R, k = i % R, rg = g * SG_ROWS + rr;
      qs[rr * RP + k] = rg < rows_total
                            ? qabs[(static_cast<size_t>(b) * rows_total + rg) * R + k]
                            : 0.f;
    }
    const int rg = g * SG_ROWS + r;
    const bool row_ok = rg < rows_total;
    const int pos_q = L - n_q + (row_ok ? rg / s.n_h : 0);
    float m = -INFINITY, l = 0.f;
    float o[SG_MAXK];
#pragma unroll
    for (int k = 0; k < SG_MAXK; ++k) o[k] = 0.f;

    for (int t = t_first; t <= t_last; ++t) {
      for (int j0 = t * p.TS; j0 < min((t + 1) * p.TS, L); j0 += SG_SUB) {
        __syncthreads();
        for (int i = tid; i < SG_SUB * R; i += SG_THREADS) {
          const int jj = i / R, k = i % R, j = j0 + jj;
          float v = 0.f;
          if (j < L) {
            int page = page_table[static_cast<size_t>(b) * max_blocks + j / s.bs];
            if (page < 0 || page >= num_blocks) {
              set_error(err, MLA_DEVERR_PAGE_RANGE);
              page = 0;
            }
            v = to_f32<T>(cache[(static_cast<size_t>(page) * s.bs + j % s.bs) * R + k]);
          }
          ks[jj * RP + k] = v;
        }
        __syncthreads();
        const int j = j0 + c16;
        float x = -INFINITY;
        if (row_ok && j < L && j <= pos_q) {
          float acc = 0.f;
          for (int k = 0; k < R; ++k) acc = fmaf(qs[r * RP + k], ks[c16 * RP + k], acc);
          x = acc * scale_log2;  // log2 domain
        }
        float mx = x;
#pragma unroll
        for (int o2 = 8; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        const float m_new = fmaxf(m, mx);
        const float pv = (x == -INFINITY) ? 0.f : exp2f(x - m_new);
        const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
        float ssum = pv;
#pragma unroll
        for (int o2 = 8; o2 > 0; o2 >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o2);
        l = l * alpha + ssum;
        m = m_new;
        ps[r * SG_SUB + c16] = pv;
        if (c16 == 0) alph[r] = alpha;
        __syncthreads();
        const float a = alph[r];
#pragma unroll
        for (int k = 0; k < SG_MAXK; ++k) {
          const int dc = c16 + 16 * k;
          if (dc < s.d_c) {
            float acc = o[k] * a;
#pragma unroll
            for (int jj = 0; jj < SG_SUB; ++jj) acc = fmaf(ps[r * SG_SUB + jj], ks[jj * RP + dc], acc);
            o[k] = acc;
          }
        }
      }
    }
    // write the partial of this piece
    if (row_ok) {
      const int slot = blockIdx.x + g * B + b;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float* dst = part_o + (static_cast<size_t>(slot) * p.RG + r) * s.d_c;
#pragma unroll
      for (int k = 0; k < SG_MAXK; ++k) {
        const int dc = c16 + 16 * k;
        if (dc < s.d_c) dst[dc] = o[k] * inv;
      }
      if (c16 == 0)
        part_lse[static_cast<size_t>(slot) * p.RG + r] =
            l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
    it = piece_end;
  }
}

template <typename T>
cudaError_t attend_simt_t(const Shape& s, const void* cache, int num_blocks,
                          const int32_t* page_table, int max_blocks, int B, int n_q,
                          const Partition& p, const WsView& ws, const int32_t* seq_lens,
                          uint32_t* err, cudaStream_t st) {
  const int RP = s.R() + 1;
  const size_t smem = sizeof(float) * (2 * 16 * RP + 16 * 16 + 16);
  auto kern = attend_simt_kernel<T>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  kern<<<p.C, SG_THREADS, smem, st>>>(s, static_cast<const T*>(cache), num_blocks, page_table,
                                      max_blocks, B, n_q, p, static_cast<const float*>(ws.qabs),
                                      ws.tiles, ws.prefix, ws.bounds, seq_lens, ws.part_o, ws.part_lse, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attend_simt(const Shape& s, mla_dtype dt, const void* cache, int num_blocks,
                               const int32_t* page_table, int max_blocks, int B, int n_q,
                               const Partition& p, const WsView& ws, const int32_t* seq_lens,
                               uint32_t* err, cudaStream_t st) {
  if (dt == MLA_F32)
    return attend_simt_t<float>(s, cache, num_blocks, page_table, max_blocks, B, n_q, p, ws,
                                seq_lens, err, st);
  return attend_simt_t<__nv_bfloat16>(s, cache, num_blocks, page_table, max_blocks, B, n_q, p,
                                      ws, seq_lens, err, st);
}

}  // namespace mla
