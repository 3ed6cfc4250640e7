// a2 (tensor-core variant): fold each head's query into latent space.
//
//   qabs[t, h, 0:512]   = W_uk[h] q_nope[t, h]       (q_lat)
//   qabs[t, h, 512:576] = RoPE(q_rope[t, h], pos_t)   (q_pe)
//
// Source: "Multi-head Latent Attention and KV Cache Compression", section
// "The absorption trick and decoupled RoPE". The content score q.(W_uk c)
// equals (W_uk^T q).c, so each query is moved into latent space once per step
// and dotted against cached latents directly. Only the position block is
// rotated, at the query's own position ("Multi-head Latent Attention: the KV
// cache, compressed", section "RoPE, and why the explanations stop here").
//
// Per head this is a dense [512 x 128] x [128 x tokens] product, so it runs on
// tcgen05: one CTA per (head, up to 128 query tokens). TMA stages the head's
// whole W_uk slice (128 KB, eight 128 x 64 boxes) and the tokens' q (three
// 3-D boxes over [token][head][dim]) into shared memory in one go, so the
// weight stream has 128 KB in flight per SM. Four threads (one per 128-row
// block of W_uk[h], each starting as soon as its two boxes have landed) issue
// 8 MMAs each with M = 128 latent rows, N = tokens, K = 128, accumulating
// q_lat^T in TMEM (4 blocks of up to 128 columns). Four warps read it back,
// one latent row per lane, and store them in bf16 (fp16 for the attention
// over an fp8 cache, whose MMAs take fp16 operands). The other four warps
// rotate q_rope meanwhile.
//
// Block (0, 0) also writes the split-KV plan (tiles per sequence, their
// prefix sum and the range boundaries), which the attention and combine
// kernels read.
#include "device_common.cuh"
#include "plan.cuh"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace mla_ptx;

constexpr int AT_TOK = 128;                    // query tokens per CTA (MMA N)
constexpr int AT_THREADS = 256;
constexpr uint32_t AT_WBOX = 128 * 128;        // 128 rows x 64 bf16
constexpr long long AT_WAIT = 2000000000LL;    // ~1 s

struct __align__(1024) AbsSmem {
  uint8_t w[8][AT_WBOX];          // box (M-block j, K-chunk kc) at index 2*j + kc
  uint8_t q[3][AT_TOK * 128];     // K-chunks 0, 1 of q_nope, then q_rope: token rows of 128 B
  uint64_t full_q, full_w[4], done;
  uint32_t tmem_base;
};

__device__ __forceinline__ uint64_t kdesc(const void* base, uint32_t byte_off) {
  return smem_desc(smem_u32(base) + byte_off, 16, 1024, kSwizzle128B);
}

template <typename OT>
__global__ void __launch_bounds__(AT_THREADS, 1)
absorb_q_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_q, Shape s,
                   const __nv_bfloat16* __restrict__ q, const uint64_t* __restrict__ rope_turns,
                   const int32_t* __restrict__ seq_lens, int B, int n_q, int max_blocks, int TS,
                   int G, int C, int K, int n_tok_box, float out_scale,
                   OT* __restrict__ qabs, int32_t* tiles, int32_t* prefix,
                   long long* bounds, int32_t* first_b, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  AbsSmem& sm = *reinterpret_cast<AbsSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const int h = blockIdx.x;
  const int t0 = blockIdx.y * AT_TOK;
  const int Tq = B * n_q;
  const int ntok = min(AT_TOK, Tq - t0);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int R = 576, DQ = 192;

  if (threadIdx.x == 0) {
    mbar_init(&sm.full_q, 1);
    for (int j = 0; j < 4; ++j) mbar_init(&sm.full_w[j], 1);
    mbar_init(&sm.done, 4);  // one commit per 128-row block
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  bool ok = true;

  // With programmatic dependent launch this CTA may start while the previous
  // kernel (the append) still runs. The packed W_uk is complete and never
  // written once its handle exists (mla_absorb_weights returns after the
  // packing kernels), so its loads start at once; the queries are read only
  // after the wait for the previous kernel.
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_q);
    for (int j = 0; j < 4; ++j) {
      mbar_arrive_expect_tx(&sm.full_w[j], 2 * AT_WBOX);
      for (int kc = 0; kc < 2; ++kc)
        tma_load_2d(sm.w[2 * j + kc], &tmap_w, 64 * kc, h * 512 + 128 * j, &sm.full_w[j]);
    }
  }
  griddep_wait();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&sm.full_q, 3 * n_tok_box * 128);
    for (int kc = 0; kc < 3; ++kc) tma_load_3d(sm.q[kc], &tmap_q, 64 * kc, h, t0, &sm.full_q);
  }
  // The attention kernel may be scheduled now; it waits for this grid to
  // complete before it reads the queries or the plan.
  griddep_launch_dependents();
  // (after the loads are on their way, so the plan costs this block no time)
  if (blockIdx.x == 0 && blockIdx.y == 0)
    write_plan<AT_THREADS>(seq_lens, B, n_q, max_blocks, s.bs, TS, G, C, K, tiles, prefix, bounds,
                           first_b, err);
  if (warp < 4 && lane == 0) {
    // block j = warp of q_lat^T, as soon as its rows of W_uk[h] are in
    const int j = warp;
    ok = mbar_wait(&sm.full_q, 0, AT_WAIT) && mbar_wait(&sm.full_w[j], 0, AT_WAIT);
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, n_tok_box, false, false);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_bf16_ss(tmem + 128 * j, kdesc(sm.w[2 * j + (k >> 2)], (k & 3) * 32),
                    kdesc(sm.q[k >> 2], (k & 3) * 32), idesc, k > 0 ? 1u : 0u);
    } else {
      set_error(err, MLA_DEVERR_TIMEOUT);
    }
    mma_commit(&sm.done);
  }

  if (warp >= 4) {
    // rotary block of each query, rotated at the query's own position, from
    // the q_rope box the TMA put in shared memory (128-byte swizzle: dims
    // [8u, 8u + 8) of token row t sit in 16-byte unit u ^ (t & 7)). Lane k
    // owns rotary pair (k, k + 32); warp w4 takes tokens w4, w4 + 4, ...
    const int k = lane, w4 = warp - 4;
    const uint64_t turns = rope_turns[k];
    const bool qok = mbar_wait(&sm.full_q, 0, AT_WAIT);
    if (!qok && k == 0) set_error(err, MLA_DEVERR_TIMEOUT);
    const uint8_t* qr = sm.q[2];
    // four tokens at a time: their loads and angle computations are
    // independent, so their latencies overlap
    constexpr int U = 4;
    for (int tb = w4; qok && tb < ntok; tb += 4 * U) {
      int pos[U];
      float x1[U], x2[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int tt = min(tb + 4 * u, ntok - 1), tok = t0 + tt;
        pos[u] = seq_lens[tok / n_q] - n_q + tok % n_q;
        const __nv_bfloat16* row = reinterpret_cast<const __nv_bfloat16*>(qr + tt * 128);
        x1[u] = __bfloat162float(row[(((k >> 3) ^ (tt & 7)) << 3) + (k & 7)]);
        x2[u] = __bfloat162float(row[((((k + 32) >> 3) ^ (tt & 7)) << 3) + (k & 7)]);
      }
      float c[U], sn[U];
#pragma unroll
      for (int u = 0; u < U; ++u) rope_cos_sin(pos[u], turns, &c[u], &sn[u]);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int tt = tb + 4 * u;
        if (tt >= ntok) break;
        OT* o = qabs + (static_cast<size_t>(t0 + tt) * s.n_h + h) * R + 512;
        o[k] = from_f32<OT>((x1[u] * c[u] - x2[u] * sn[u]) * out_scale);
        o[k + 32] = from_f32<OT>((x1[u] * sn[u] + x2[u] * c[u]) * out_scale);
      }
    }
  } else {
    // q_lat^T from TMEM (lane = latent row inside M-block j, column =
    // token), transposed through shared memory: the MMAs are done with
    // W_uk[h], so its buffer holds q_lat as [token][512]; then every token's
    // 1 KB row goes out in 16-byte stores.
    const bool done = mbar_wait(&sm.done, 0, 2 * AT_WAIT);
    tc_fence_after();
    if (!done) {
      if (lane == 0 && warp == 0) set_error(err, MLA_DEVERR_TIMEOUT);
    } else {
      OT* stg = reinterpret_cast<OT*>(sm.w[0]);  // [n_tok_box][512]
      const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
      // 16 tokens of all four blocks per TMEM round trip
      for (int c0 = 0; c0 < n_tok_box; c0 += 16) {
        float v[4][16];
#pragma unroll
        for (int j = 0; j < 4; ++j) tmem_ld16(tmem + lane_base + 128 * j + c0, v[j]);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int dc = 128 * j + 32 * warp + lane;
#pragma unroll
          for (int i = 0; i < 16; ++i) stg[(c0 + i) * 512 + dc] = from_f32<OT>(v[j][i] * out_scale);
        }
      }
    }
    named_bar_sync(1, 128);  // the four warps' rows are in place
    if (done) {
      const OT* stg = reinterpret_cast<const OT*>(sm.w[0]);
      for (int i = threadIdx.x; i < ntok * 64; i += 128) {
        const int tt = i / 64, u = i % 64;  // 16-byte unit u of token tt's 512 values
        *reinterpret_cast<uint4*>(qabs + (static_cast<size_t>(t0 + tt) * s.n_h + h) * R + 8 * u) =
            *reinterpret_cast<const uint4*>(stg + tt * 512 + 8 * u);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}


template <typename OT>
cudaError_t absorb_q_tc_t(const Shape& s, const Weights* w, const void* q,
                          const int32_t* seq_lens, int max_blocks, int B, int n_q,
                          const Partition& p, const WsView& ws, float out_scale, uint32_t* err,
                          cudaStream_t st) {
  const int Tq = B * n_q;
  const int n_tok_box = min(AT_TOK, ((Tq + 15) / 16) * 16);
  TmapSpec ws_spec{};
  ws_spec.dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  ws_spec.rank = 2;
  ws_spec.base = w->w_uk;
  ws_spec.dims[0] = 128;
  ws_spec.dims[1] = static_cast<uint64_t>(s.n_h) * 512;
  ws_spec.strides[0] = 256;
  ws_spec.box[0] = 64;
  ws_spec.box[1] = 128;
  ws_spec.swizzle = CU_TENSOR_MAP_SWIZZLE_128B;
  TmapSpec qs{};
  qs.dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  qs.rank = 3;
  qs.base = q;
  qs.dims[0] = 192;
  qs.dims[1] = s.n_h;
  qs.dims[2] = Tq;
  qs.strides[0] = 192 * 2;
  qs.strides[1] = static_cast<uint64_t>(s.n_h) * 192 * 2;
  qs.box[0] = 64;
  qs.box[1] = 1;
  qs.box[2] = n_tok_box;
  qs.swizzle = CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap tw, tq;
  if (!get_tmap(ws_spec, &tw) || !get_tmap(qs, &tq)) return cudaErrorInvalidValue;
  const size_t smem = sizeof(AbsSmem) + 1024;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(absorb_q_tc_kernel<OT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.n_h, (Tq + AT_TOK - 1) / AT_TOK, 1);
  cfg.blockDim = dim3(AT_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // may start while the previous kernel finishes (see the kernel's wait)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, absorb_q_tc_kernel<OT>,
      tw, tq, s, static_cast<const __nv_bfloat16*>(q), w->rope_turns, seq_lens, B, n_q, max_blocks,
      p.TS, p.G, p.C, p.K, n_tok_box, out_scale, static_cast<OT*>(ws.qabs), ws.tiles,
      ws.prefix, ws.bounds, ws.first_b, err);
}

}  // namespace

bool absorb_tc_supported(const Shape& s, mla_dtype dt) {
  return dt == MLA_BF16 && s.d_c == 512 && s.d_nope == 128 && s.d_r == 64;
}

cudaError_t launch_absorb_q_tc(const Shape& s, const Weights* w, const void* q,
                               const int32_t* seq_lens, int max_blocks, int B, int n_q,
                               const Partition& p, const WsView& ws, float out_scale,
                               bool q_half, uint32_t* err, cudaStream_t st) {
  if (q_half)
    return absorb_q_tc_t<__half>(s, w, q, seq_lens, max_blocks, B, n_q, p, ws, out_scale, err,
                                 st);
  return absorb_q_tc_t<__nv_bfloat16>(s, w, q, seq_lens, max_blocks, B, n_q, p, ws, out_scale,
                                      err, st);
}

}  // namespace mla
