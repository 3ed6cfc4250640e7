// a4 + a5: merge the split-KV partials with their log-sum-exps, then
// up-project the latent output through W_uv.
//
//   lse   = log sum_s exp(lse_s)
//   o_lat = sum_s exp(lse_s - lse) * o_s          (o_s already divided by l_s)
//   out   = o_lat W_uv[h]
//
// The value-side up-projection is applied after the weighted sum, once per
// head and query, instead of to every cached token. Source: "Multi-head
// Latent Attention and KV Cache Compression", section "The absorption trick
// and decoupled RoPE" (the value up-projection is absorbed on the output
// side the same way W_uk is on the query side).
//
// One CTA per (head, tile of 16 query tokens). It reads that head's
// [d_c x d_v] slice of W_uv once and reuses it for all 16 tokens.
#include <cmath>

#include "device_common.cuh"

namespace mla {
namespace {

constexpr int CB_TOK = 16, CB_THREADS = 128;

template <typename T>
__global__ void __launch_bounds__(CB_THREADS)
combine_kernel(Shape s, const T* __restrict__ w_uv, const int32_t* __restrict__ tiles,
               const int32_t* __restrict__ prefix, int B, int n_q, Partition p,
               const float* __restrict__ part_o, const float* __restrict__ part_lse,
               float* __restrict__ out) {
  extern __shared__ float olat[];  // [CB_TOK][d_c]
  __shared__ int c_lo[CB_TOK], c_hi[CB_TOK], row_off[CB_TOK];
  __shared__ float m_max[CB_TOK], inv_den[CB_TOK];
  const int h = blockIdx.x, tok0 = blockIdx.y * CB_TOK;
  const int Tq = B * n_q, ntok = min(CB_TOK, Tq - tok0);
  const long long T_all = prefix[B];
  const long long N = T_all * p.G;

  // 1. per token: the CTAs holding its pieces, the max lse and the normaliser
  if (threadIdx.x < CB_TOK) {
    const int t = threadIdx.x;
    int c0 = 0, c1 = -1, off = 0;
    float M = -INFINITY, den = 0.f;
    if (t < ntok) {
      const int tok = tok0 + t, b = tok / n_q, qi = tok % n_q;
      const int r = qi * s.n_h + h, g = r / p.RG, rr = r % p.RG;
      off = (g * B + b) * p.RG + rr;  // slot (c + g*B + b) * RG + rr = c*RG + off
      if (tiles[b] > 0) {
        const long long first = g * T_all + prefix[b], last = first + tiles[b] - 1;
        c0 = cta_of_item(first, N, p.C);
        c1 = cta_of_item(last, N, p.C);
        for (int c = c0; c <= c1; ++c) {
          if (range_begin(c, N, p.C) == range_begin(c + 1, N, p.C)) continue;
          M = fmaxf(M, part_lse[static_cast<size_t>(c) * p.RG + off]);
        }
        if (M != -INFINITY) {
          for (int c = c0; c <= c1; ++c) {
            if (range_begin(c, N, p.C) == range_begin(c + 1, N, p.C)) continue;
            den += expf(part_lse[static_cast<size_t>(c) * p.RG + off] - M);
          }
        }
      }
    }
    c_lo[t] = c0;
    c_hi[t] = (M == -INFINITY) ? -1 : c1;
    row_off[t] = off;
    m_max[t] = M;
    inv_den[t] = den > 0.f ? 1.f / den : 0.f;
  }
  __syncthreads();
  // 2. o_lat = weighted sum of the normalised partials
  for (int t = 0; t < CB_TOK; ++t) {
    for (int dc = threadIdx.x; dc < s.d_c; dc += CB_THREADS) {
      float acc = 0.f;
      for (int c = c_lo[t]; c <= c_hi[t]; ++c) {
        if (range_begin(c, N, p.C) == range_begin(c + 1, N, p.C)) continue;
        const size_t row = static_cast<size_t>(c) * p.RG + row_off[t];
        const float w = expf(part_lse[row] - m_max[t]) * inv_den[t];
        acc = fmaf(w, part_o[row * s.d_c + dc], acc);
      }
      olat[t * s.d_c + dc] = acc;
    }
  }
  __syncthreads();
  // 3. out = o_lat W_uv[h]
  const T* W = w_uv + static_cast<size_t>(h) * s.d_c * s.d_v;
  for (int dv = threadIdx.x; dv < s.d_v; dv += CB_THREADS) {
    float acc[CB_TOK];
#pragma unroll
    for (int t = 0; t < CB_TOK; ++t) acc[t] = 0.f;
    for (int dc = 0; dc < s.d_c; ++dc) {
      const float w = to_f32<T>(W[static_cast<size_t>(dc) * s.d_v + dv]);
#pragma unroll
      for (int t = 0; t < CB_TOK; ++t) acc[t] = fmaf(olat[t * s.d_c + dc], w, acc[t]);
    }
    for (int t = 0; t < ntok; ++t)
      out[(static_cast<size_t>(tok0 + t) * s.n_h + h) * s.d_v + dv] = acc[t];
  }
}

template <typename T>
cudaError_t combine_t(const Shape& s, const Weights* w, int B, int n_q, const Partition& p,
                      const WsView& ws, float* out, cudaStream_t st) {
  const int Tq = B * n_q;
  dim3 grid(s.n_h, (Tq + CB_TOK - 1) / CB_TOK);
  const size_t smem = sizeof(float) * CB_TOK * s.d_c;
  auto kern = combine_kernel<T>;
  if (smem > 40 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  kern<<<grid, CB_THREADS, smem, st>>>(s, static_cast<const T*>(w->w_uv), ws.tiles, ws.prefix, B,
                                       n_q, p, ws.part_o, ws.part_lse, out);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const Shape& s, mla_dtype dt, const Weights* w,
                           const int32_t* seq_lens, int B, int n_q, const Partition& p,
                           const WsView& ws, float* out, cudaStream_t st) {
  (void)seq_lens;
  if (dt == MLA_F32) return combine_t<float>(s, w, B, n_q, p, ws, out, st);
  return combine_t<__nv_bfloat16>(s, w, B, n_q, p, ws, out, st);
}

}  // namespace mla
