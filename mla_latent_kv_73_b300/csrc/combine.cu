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
// table rb[0..C] of the attention partition, then the merge weights
// [CB_TOK][C + 1].
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
  float* wts = reinterpret_cast<float*>(rb + p.C + 1);  // [CB_TOK][C+1]
  __shared__ int c_lo[CB_TOK], c_hi[CB_TOK], row_off[CB_TOK];
  const int h = blockIdx.x, tok0 = blockIdx.y * CB_TOK;
  const int Tq = B * n_q, ntok = min(CB_TOK, Tq - tok0);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // 1. per token: the ranges holding its pieces and their merge weights
  //    exp(lse_s - lse). The plan loads of all tokens go out together; then
  //    half a warp per token, its lanes taking the pieces, loads the lse
  //    values.
  const long long T_all = prefix[B];
  for (int c = threadIdx.x; c <= p.C; c += CB_THREADS) rb[c] = bounds[c];  // all 0 without tiles
  int my_tiles = 0, my_off = 0;
  long long my_first = 0;
  if (threadIdx.x < ntok) {
    const int tok = tok0 + threadIdx.x, b = tok / n_q, qi = tok % n_q;
    const int r = qi * s.n_h + h, g = r / p.RG, rr = r % p.RG;
    my_off = (g * B + b) * p.RG + rr;  // row of slot (c + g*B + b) is c*RG + off
    my_tiles = tiles[b];
    my_first = static_cast<long long>(g) * T_all + prefix[b];
  }
  __syncthreads();  // range starts in place
  if (threadIdx.x < CB_TOK) {
    int c0 = 0, c1 = -1;
    if (my_tiles > 0) {
      c0 = range_of_item(rb, p.C, my_first);
      c1 = range_of_item(rb, p.C, my_first + my_tiles - 1);
    }
    c_lo[threadIdx.x] = c0;
    c_hi[threadIdx.x] = c1;
    row_off[threadIdx.x] = my_off;
  }
  __syncthreads();
  for (int tb = 0; tb < ntok; tb += 2 * (CB_THREADS / 32)) {
    const int t = tb + 2 * warp + (lane >> 4), hl = lane & 15;
    const bool live = t < ntok;
    const int c0 = live ? c_lo[t] : 0, c1 = live ? c_hi[t] : -1;
    const int off = live ? row_off[t] : 0;
    float M = -INFINITY;
    for (int c = c0 + hl; c <= c1; c += 16) {
      const float x = rb[c] != rb[c + 1] ? part_lse[static_cast<size_t>(c) * p.RG + off] : -INFINITY;
      wts[t * (p.C + 1) + (c - c0)] = x;
      M = fmaxf(M, x);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float den = 0.f;
    for (int c = c0 + hl; c <= c1; c += 16) {
      const float e = M == -INFINITY ? 0.f : expf(wts[t * (p.C + 1) + (c - c0)] - M);
      wts[t * (p.C + 1) + (c - c0)] = e;
      den += e;
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int c = c0 + hl; c <= c1; c += 16) wts[t * (p.C + 1) + (c - c0)] *= inv;
    if (live && hl == 0 && M == -INFINITY) c_hi[t] = -1;  // no piece holds a visible token
  }
  __syncthreads();

  // 2. o_lat = weighted sum of the normalised partials. A thread owns four
  //    latent dims (one 16-byte load per piece) of several tokens; pieces of
  //    empty ranges carry weight 0 and are not read.
  const int d4 = s.d_c / 4;  // d_c % 4 == 0
  for (int i = threadIdx.x; i < CB_TOK * d4; i += CB_THREADS) {
    const int t = i / d4, dc = 4 * (i % d4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < ntok) {
      const int c0 = c_lo[t], c1 = c_hi[t];
      const float* w = wts + t * (p.C + 1) - c0;
#pragma unroll 4
      for (int c = c0; c <= c1; ++c) {
        const float wc = w[c];
        if (wc == 0.f) continue;
        const float4 v = *reinterpret_cast<const float4*>(
            part_o + (static_cast<size_t>(c) * p.RG + row_off[t]) * s.d_c + dc);
        acc.x = fmaf(wc, v.x, acc.x);
        acc.y = fmaf(wc, v.y, acc.y);
        acc.z = fmaf(wc, v.z, acc.z);
        acc.w = fmaf(wc, v.w, acc.w);
      }
      if (olat_out) {  // latent mode: o_lat [B*n_q][n_h*d_c], no up-projection
        *reinterpret_cast<float4*>(olat_out + (static_cast<size_t>(tok0 + t) * s.n_h + h) * s.d_c +
                                   dc) = acc;
        continue;
      }
    }
    if (!olat_out) {
      olat[(dc + 0) * CB_TOK + t] = acc.x;
      olat[(dc + 1) * CB_TOK + t] = acc.y;
      olat[(dc + 2) * CB_TOK + t] = acc.z;
      olat[(dc + 3) * CB_TOK + t] = acc.w;
    }
  }
  if (olat_out) return;
  __syncthreads();

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
                      sizeof(long long) * (p.C + 1) + sizeof(float) * CB_TOK * (p.C + 1);
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
