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
// One CTA per (head, tile of 16 query tokens). It streams that head's
// [d_v x d_c] slice of W_uv once with 16-byte loads and reuses each element
// for all 16 tokens. In latent mode (the full-fold layer, whose output
// projection has W_uv folded in) it writes o_lat instead and stops there.
#include <cmath>

#include "device_common.cuh"
#include "plan.cuh"

namespace mla {
namespace {

constexpr int CB_TOK = 16, CB_THREADS = 256;

// Dynamic shared memory: o_lat [d_c][CB_TOK] (token fastest), then the
// partial outputs of the two d_c halves [2][CB_TOK][d_v], then the range
// table rb[0..C] of the attention partition.
template <typename T>
__global__ void __launch_bounds__(CB_THREADS)
combine_kernel(Shape s, const T* __restrict__ w_uv, const int32_t* __restrict__ tiles,
               const int32_t* __restrict__ prefix, const long long* __restrict__ bounds, int B,
               int n_q, Partition p,
               const float* __restrict__ part_o, const float* __restrict__ part_lse,
               float* __restrict__ out, float* __restrict__ olat_out) {
  extern __shared__ __align__(16) float sm[];
  float* olat = sm;                                   // [d_c][CB_TOK]
  float* half_out = olat + s.d_c * CB_TOK;            // [2][CB_TOK][d_v]
  long long* rb = reinterpret_cast<long long*>(half_out + 2 * CB_TOK * s.d_v);  // [C+1]
  __shared__ int c_lo[CB_TOK], c_hi[CB_TOK], row_off[CB_TOK];
  __shared__ float m_max[CB_TOK], inv_den[CB_TOK];
  const int h = blockIdx.x, tok0 = blockIdx.y * CB_TOK;
  const int Tq = B * n_q, ntok = min(CB_TOK, Tq - tok0);
  const long long T_all = prefix[B];
  const long long N = T_all * p.G;

  for (int c = threadIdx.x; c <= p.C; c += CB_THREADS) rb[c] = N > 0 ? bounds[c] : 0;
  __syncthreads();

  // 1. per token: the CTAs holding its pieces, the max lse and the normaliser
  if (threadIdx.x < CB_TOK) {
    const int t = threadIdx.x;
    int c0 = 0, c1 = -1, off = 0;
    float M = -INFINITY, den = 0.f;
    if (t < ntok) {
      const int tok = tok0 + t, b = tok / n_q, qi = tok % n_q;
      const int r = qi * s.n_h + h, g = r / p.RG, rr = r % p.RG;
      off = (g * B + b) * p.RG + rr;  // row of slot (c + g*B + b) is c*RG + off
      if (tiles[b] > 0) {
        const long long first = g * T_all + prefix[b], last = first + tiles[b] - 1;
        c0 = range_of_item(rb, p.C, first);
        c1 = range_of_item(rb, p.C, last);
        for (int c = c0; c <= c1; ++c)
          if (rb[c] != rb[c + 1]) M = fmaxf(M, part_lse[static_cast<size_t>(c) * p.RG + off]);
        if (M != -INFINITY)
          for (int c = c0; c <= c1; ++c)
            if (rb[c] != rb[c + 1]) den += expf(part_lse[static_cast<size_t>(c) * p.RG + off] - M);
      }
    }
    c_lo[t] = c0;
    c_hi[t] = (M == -INFINITY) ? -1 : c1;
    row_off[t] = off;
    m_max[t] = M;
    inv_den[t] = den > 0.f ? 1.f / den : 0.f;
  }
  __syncthreads();

  // 2. o_lat = weighted sum of the normalised partials (coalesced over d_c)
  for (int t = 0; t < CB_TOK; ++t) {
    for (int dc = threadIdx.x; dc < s.d_c; dc += CB_THREADS) {
      float acc = 0.f;
      for (int c = c_lo[t]; c <= c_hi[t]; ++c) {
        if (rb[c] == rb[c + 1]) continue;
        const size_t row = static_cast<size_t>(c) * p.RG + row_off[t];
        acc = fmaf(expf(part_lse[row] - m_max[t]) * inv_den[t], part_o[row * s.d_c + dc], acc);
      }
      olat[dc * CB_TOK + t] = acc;
    }
  }
  __syncthreads();
  if (olat_out) {  // latent mode: o_lat [B*n_q][n_h*d_c], no up-projection
    for (int i = threadIdx.x; i < ntok * s.d_c; i += CB_THREADS) {
      const int t = i / s.d_c, dc = i % s.d_c;
      olat_out[(static_cast<size_t>(tok0 + t) * s.n_h + h) * s.d_c + dc] = olat[dc * CB_TOK + t];
    }
    return;
  }

  // 3. out = o_lat W_uv[h]: W_uv is packed [h][d_v][d_c]. A thread owns one
  // output column for all 16 tokens and half of the d_c reduction.
  constexpr int V = Vec<T>::N;
  const T* W = w_uv + static_cast<size_t>(h) * s.d_v * s.d_c;
  const int dc_half = (s.d_c + 1) / 2;
  const bool vec_ok = s.d_c % (2 * V) == 0;
  for (int idx = threadIdx.x; idx < 2 * s.d_v; idx += CB_THREADS) {
    const int dv = idx % s.d_v, part = idx / s.d_v;
    const int k0 = part * dc_half, k1 = min(s.d_c, k0 + dc_half);
    float acc[CB_TOK];
#pragma unroll
    for (int t = 0; t < CB_TOK; ++t) acc[t] = 0.f;
    const T* wr = W + static_cast<size_t>(dv) * s.d_c;
    if (vec_ok) {
#pragma unroll 2
      for (int k = k0; k < k1; k += V) {
        float wv[V];
        load_vec<T>(wr + k, wv);
#pragma unroll
        for (int j = 0; j < V; ++j) {
          const float4* ov = reinterpret_cast<const float4*>(olat + (k + j) * CB_TOK);
#pragma unroll
          for (int u = 0; u < CB_TOK / 4; ++u) {
            const float4 x = ov[u];
            acc[4 * u + 0] = fmaf(wv[j], x.x, acc[4 * u + 0]);
            acc[4 * u + 1] = fmaf(wv[j], x.y, acc[4 * u + 1]);
            acc[4 * u + 2] = fmaf(wv[j], x.z, acc[4 * u + 2]);
            acc[4 * u + 3] = fmaf(wv[j], x.w, acc[4 * u + 3]);
          }
        }
      }
    } else {
      for (int k = k0; k < k1; ++k) {
        const float wv = to_f32<T>(wr[k]);
#pragma unroll
        for (int t = 0; t < CB_TOK; ++t) acc[t] = fmaf(wv, olat[k * CB_TOK + t], acc[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < CB_TOK; ++t) half_out[(part * CB_TOK + t) * s.d_v + dv] = acc[t];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < ntok * s.d_v; i += CB_THREADS) {
    const int t = i / s.d_v, dv = i % s.d_v;
    out[(static_cast<size_t>(tok0 + t) * s.n_h + h) * s.d_v + dv] =
        half_out[t * s.d_v + dv] + half_out[(CB_TOK + t) * s.d_v + dv];
  }
}

template <typename T>
cudaError_t combine_t(const Shape& s, const T* w_uv, int B, int n_q, const Partition& p,
                      const WsView& ws, float* out, float* olat, cudaStream_t st) {
  const int Tq = B * n_q;
  dim3 grid(s.n_h, (Tq + CB_TOK - 1) / CB_TOK);
  const size_t smem = sizeof(float) * (CB_TOK * s.d_c + 2 * CB_TOK * s.d_v) +
                      sizeof(long long) * (p.C + 1);
  auto kern = combine_kernel<T>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  kern<<<grid, CB_THREADS, smem, st>>>(s, w_uv, ws.tiles, ws.prefix, ws.bounds, B, n_q, p,
                                       ws.part_o, ws.part_lse, out, olat);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const Shape& s, mla_dtype dt, const Weights* w,
                           const int32_t* seq_lens, int B, int n_q, const Partition& p,
                           const WsView& ws, float* out, cudaStream_t st) {
  (void)seq_lens;
  if (dt == MLA_F32)
    return combine_t<float>(s, static_cast<const float*>(w->w_uv), B, n_q, p, ws, out, nullptr,
                            st);
  return combine_t<__nv_bfloat16>(s, static_cast<const __nv_bfloat16*>(w->w_uv), B, n_q, p, ws,
                                  out, nullptr, st);
}

cudaError_t launch_combine_latent(const Shape& s, int B, int n_q, const Partition& p,
                                  const WsView& ws, float* olat, cudaStream_t st) {
  return combine_t<float>(s, nullptr, B, n_q, p, ws, nullptr, olat, st);
}

}  // namespace mla
