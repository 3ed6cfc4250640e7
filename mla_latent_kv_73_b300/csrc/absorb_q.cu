// a2: fold each head's query into latent space, and plan the split-KV work.
//
//   qabs[t, h, 0:d_c]    = W_uk[h] q_nope[t, h]        (q_lat, d_c wide)
//   qabs[t, h, d_c:d_c+d_r] = RoPE(q_rope[t, h], pos_t)
//
// Source: "Multi-head Latent Attention and KV Cache Compression", section
// "The absorption trick and decoupled RoPE". The score q.k_j with
// k_j = W_u c_j equals (W_u^T q).c_j, so the query is moved into latent
// space once and dotted against cached latents directly. Only the position
// block is rotated, per query position ("Multi-head Latent Attention: the
// KV cache, compressed", section "RoPE, and why the explanations stop here").
//
// The queries are stored in the cache dtype for the tensor-core attention
// (its MMA operands) and in fp32 for the CUDA-core attention, which then
// keeps every score in fp32 from the query on.
//
// One CTA per (head, tile of 16 query tokens). It streams that head's
// [d_c x d_nope] slice of W_uk once with 16-byte loads. Each thread owns two
// latent rows and all 16 tokens, so every weight element is read once.
//
// Block (0, 0) also writes the split-KV plan: the tiles of each sequence,
// their prefix sum and the range boundaries. The attention and combine
// kernels both read it.
#include "device_common.cuh"
#include "plan.cuh"

namespace mla {
namespace {

constexpr int AQ_TOK = 16, AQ_THREADS = 256;

template <typename T, typename QT>
__global__ void __launch_bounds__(AQ_THREADS)
absorb_q_kernel(Shape s, const T* __restrict__ q, const T* __restrict__ w_uk,
                const uint64_t* __restrict__ rope_turns, const int32_t* __restrict__ seq_lens, int B,
                int n_q, int max_blocks, int TS, int G, int C, int K, float out_scale,
                QT* __restrict__ qabs, int32_t* tiles, int32_t* prefix, long long* bounds,
                int32_t* first_b, uint32_t* err) {
  extern __shared__ __align__(16) float qn[];  // [d_nope][AQ_TOK], token fastest
  const int h = blockIdx.x;
  const int tok0 = blockIdx.y * AQ_TOK;
  const int Tq = B * n_q;
  const int dq = s.d_nope + s.d_r, R = s.R();
  if (blockIdx.x == 0 && blockIdx.y == 0)
    write_plan<AQ_THREADS>(seq_lens, B, n_q, max_blocks, s.bs, TS, G, C, K, tiles, prefix, bounds,
                           first_b, err);

  const int ntok = min(AQ_TOK, Tq - tok0);
  for (int i = threadIdx.x; i < AQ_TOK * s.d_nope; i += AQ_THREADS) {
    const int t = i / s.d_nope, n = i % s.d_nope;
    qn[n * AQ_TOK + t] =
        t < ntok ? to_f32<T>(q[(static_cast<size_t>(tok0 + t) * s.n_h + h) * dq + n]) : 0.f;
  }
  __syncthreads();

  // Two latent rows per thread; the 16 token values of each n are one
  // broadcast shared-memory read of 4 float4.
  constexpr int V = Vec<T>::N;
  const T* W = w_uk + static_cast<size_t>(h) * s.d_c * s.d_nope;
  const bool vec_ok = s.d_nope % V == 0;
  for (int dc0 = 2 * threadIdx.x; dc0 < s.d_c; dc0 += 2 * AQ_THREADS) {
    const bool two = dc0 + 1 < s.d_c;
    float acc0[AQ_TOK], acc1[AQ_TOK];
#pragma unroll
    for (int t = 0; t < AQ_TOK; ++t) acc0[t] = acc1[t] = 0.f;
    const T* r0 = W + static_cast<size_t>(dc0) * s.d_nope;
    const T* r1 = two ? r0 + s.d_nope : r0;
    if (vec_ok) {
#pragma unroll 2
      for (int n0 = 0; n0 < s.d_nope; n0 += V) {
        float w0[V], w1[V];
        load_vec<T>(r0 + n0, w0);
        load_vec<T>(r1 + n0, w1);
#pragma unroll
        for (int j = 0; j < V; ++j) {
          const float4* qv = reinterpret_cast<const float4*>(qn + (n0 + j) * AQ_TOK);
#pragma unroll
          for (int u = 0; u < AQ_TOK / 4; ++u) {
            const float4 x = qv[u];
            acc0[4 * u + 0] = fmaf(w0[j], x.x, acc0[4 * u + 0]);
            acc0[4 * u + 1] = fmaf(w0[j], x.y, acc0[4 * u + 1]);
            acc0[4 * u + 2] = fmaf(w0[j], x.z, acc0[4 * u + 2]);
            acc0[4 * u + 3] = fmaf(w0[j], x.w, acc0[4 * u + 3]);
            acc1[4 * u + 0] = fmaf(w1[j], x.x, acc1[4 * u + 0]);
            acc1[4 * u + 1] = fmaf(w1[j], x.y, acc1[4 * u + 1]);
            acc1[4 * u + 2] = fmaf(w1[j], x.z, acc1[4 * u + 2]);
            acc1[4 * u + 3] = fmaf(w1[j], x.w, acc1[4 * u + 3]);
          }
        }
      }
    } else {
      for (int n = 0; n < s.d_nope; ++n) {
        const float w0 = to_f32<T>(r0[n]), w1 = to_f32<T>(r1[n]);
#pragma unroll
        for (int t = 0; t < AQ_TOK; ++t) {
          acc0[t] = fmaf(w0, qn[n * AQ_TOK + t], acc0[t]);
          acc1[t] = fmaf(w1, qn[n * AQ_TOK + t], acc1[t]);
        }
      }
    }
    for (int t = 0; t < ntok; ++t) {
      QT* o = qabs + (static_cast<size_t>(tok0 + t) * s.n_h + h) * R + dc0;
      o[0] = from_f32<QT>(acc0[t] * out_scale);
      if (two) o[1] = from_f32<QT>(acc1[t] * out_scale);
    }
  }

  // rotary block of the query, rotated at the query's own position
  const int half = s.d_r / 2;
  for (int i = threadIdx.x; i < ntok * half; i += AQ_THREADS) {
    const int t = i / half, k = i % half;
    const int tok = tok0 + t, b = tok / n_q, qi = tok % n_q;
    const int pos = seq_lens[b] - n_q + qi;
    const T* qr = q + (static_cast<size_t>(tok) * s.n_h + h) * dq + s.d_nope;
    const float x1 = to_f32<T>(qr[k]), x2 = to_f32<T>(qr[k + half]);
    float c, sn;
    rope_cos_sin(pos, rope_turns[k], &c, &sn);
    QT* o = qabs + (static_cast<size_t>(tok) * s.n_h + h) * R + s.d_c;
    o[k] = from_f32<QT>((x1 * c - x2 * sn) * out_scale);
    o[k + half] = from_f32<QT>((x1 * sn + x2 * c) * out_scale);
  }
}

template <typename T, typename QT>
cudaError_t absorb_q_t(const Shape& s, const Weights* w, const void* q, const int32_t* seq_lens,
                       int max_blocks, int B, int n_q, const Partition& p, const WsView& ws,
                       float out_scale, uint32_t* err, cudaStream_t st) {
  const int Tq = B * n_q;
  dim3 grid(s.n_h, (Tq + AQ_TOK - 1) / AQ_TOK);
  const size_t smem = sizeof(float) * AQ_TOK * s.d_nope;  // up to 64 KB (d_nope <= 1024)
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(absorb_q_kernel<T, QT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  absorb_q_kernel<T, QT><<<grid, AQ_THREADS, smem, st>>>(
      s, static_cast<const T*>(q), static_cast<const T*>(w->w_uk), w->rope_turns, seq_lens, B, n_q,
      max_blocks, p.TS, p.G, p.C, p.K, out_scale, static_cast<QT*>(ws.qabs), ws.tiles, ws.prefix,
      ws.bounds, ws.first_b, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_absorb_q(const Shape& s, mla_dtype dt, const Weights* w, const void* q,
                            const int32_t* seq_lens, int max_blocks, int B, int n_q,
                            const Partition& p, const WsView& ws, float out_scale, bool q_f32,
                            uint32_t* err, cudaStream_t st) {
  if (dt == MLA_F32)
    return absorb_q_t<float, float>(s, w, q, seq_lens, max_blocks, B, n_q, p, ws, out_scale, err,
                                    st);
  if (q_f32)
    return absorb_q_t<__nv_bfloat16, float>(s, w, q, seq_lens, max_blocks, B, n_q, p, ws,
                                            out_scale, err, st);
  return absorb_q_t<__nv_bfloat16, __nv_bfloat16>(s, w, q, seq_lens, max_blocks, B, n_q, p, ws,
                                                  out_scale, err, st);
}

}  // namespace mla
