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
// tcgen05: one CTA per (head, slice of the query tokens). TMA stages the
// head's whole W_uk slice (128 KB, eight 128 x 64 boxes) once, so the weight
// stream has 128 KB in flight per SM, and the tokens' q (three 3-D boxes over
// [token][head][dim]) 64 tokens at a time into two buffers. Per sub-block of
// 64 tokens, four threads (one per 128-row block of W_uk[h], the first time
// as soon as its two boxes have landed) issue 8 MMAs each with M = 128 latent
// rows, N = tokens, K = 128, accumulating q_lat^T in one of two TMEM buffers
// (4 blocks of 64 columns each). Four warps read it back, one latent row per
// lane, and store them in bf16 (fp16 for the attention over an fp8 cache,
// whose MMAs take fp16 operands). The other four warps rotate q_rope
// meanwhile. Decode batches of up to 64 queries are one sub-block.
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

constexpr int AT_SB = 64;                      // query tokens per sub-block (MMA N)
constexpr int AT_THREADS = 256;
constexpr uint32_t AT_WBOX = 128 * 128;        // 128 rows x 64 bf16
constexpr long long AT_WAIT = 2000000000LL;    // ~1 s
constexpr int AT_STG_TOK = 16;                 // tokens per epilogue staging round

template <typename OT>
struct __align__(1024) AbsSmem {
  uint8_t w[8][AT_WBOX];              // box (M-block j, K-chunk kc) at index 2*j + kc
  uint8_t q[2][3][AT_SB * 128];       // [buffer][q_nope K-chunk 0, 1, q_rope]: token rows of 128 B
  OT stg[AT_STG_TOK][512];            // q_lat rows on their way out
  uint64_t full_w[4], full_q[2], mma_done[2], tmem_free[2];
  uint32_t tmem_base;
};

__device__ __forceinline__ uint64_t kdesc(const void* base, uint32_t byte_off) {
  return smem_desc(smem_u32(base) + byte_off, 16, 1024, kSwizzle128B);
}

// One CTA per (head, slice of the query tokens). The head's W_uk stays in
// shared memory while the CTA walks its sub-blocks of 64 tokens (blockIdx.y,
// blockIdx.y + gridDim.y, ...); the queries and the TMEM accumulator are
// double-buffered, so the MMAs of a sub-block overlap the epilogue of the one
// before and the loads of the one after.
//   warps 0-3: lane 0 of warp j issues block j's MMAs; all four read q_lat^T
//              back (one latent row per lane) and store it
//   warps 4-7: rotate q_rope; thread 128 loads W_uk and the queries
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
  AbsSmem<OT>& sm = *reinterpret_cast<AbsSmem<OT>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                    ~static_cast<uintptr_t>(1023));
  const int h = blockIdx.x;
  const int Tq = B * n_q;
  const int n_sb = (Tq + AT_SB - 1) / AT_SB;
  // sub-blocks of this CTA: sb_i = blockIdx.y + i * gridDim.y, i < my_n
  const int my_n = blockIdx.y < n_sb ? (n_sb - 1 - blockIdx.y) / gridDim.y + 1 : 0;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int R = 576;
  const uint32_t q_tx = 3 * n_tok_box * 128;

  if (threadIdx.x == 0) {
    for (int j = 0; j < 4; ++j) mbar_init(&sm.full_w[j], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.full_q[b], 1);
      mbar_init(&sm.mma_done[b], 4);   // one commit per 128-row block
      mbar_init(&sm.tmem_free[b], 4);  // one arrival per epilogue warp
    }
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

  // With programmatic dependent launch this CTA may start while the previous
  // kernel (the append) still runs. The packed W_uk is complete and never
  // written once its handle exists (mla_absorb_weights returns after the
  // packing kernels), so its loads start at once; the queries are read only
  // after the wait for the previous kernel.
  if (threadIdx.x == 128 && my_n > 0) {
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_q);
    for (int j = 0; j < 4; ++j) {
      mbar_arrive_expect_tx(&sm.full_w[j], 2 * AT_WBOX);
      for (int kc = 0; kc < 2; ++kc)
        tma_load_2d(sm.w[2 * j + kc], &tmap_w, 64 * kc, h * 512 + 128 * j, &sm.full_w[j]);
    }
  }
  griddep_wait();
  if (threadIdx.x == 128) {
    for (int i = 0; i < my_n && i < 2; ++i) {
      const int t0 = (blockIdx.y + i * gridDim.y) * AT_SB;
      mbar_arrive_expect_tx(&sm.full_q[i], q_tx);
      for (int kc = 0; kc < 3; ++kc)
        tma_load_3d(sm.q[i][kc], &tmap_q, 64 * kc, h, t0, &sm.full_q[i]);
    }
  }
  // The attention kernel may be scheduled now; it waits for this grid to
  // complete before it reads the queries or the plan.
  griddep_launch_dependents();
  // (after the loads are on their way, so the plan costs this block no time)
  if (blockIdx.x == 0 && blockIdx.y == 0)
    write_plan<AT_THREADS>(seq_lens, B, n_q, max_blocks, s.bs, TS, G, C, K, tiles, prefix, bounds,
                           first_b, err);

  bool ok = true;
  if (warp < 4) {
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    const uint32_t idesc = idesc_bf16_f32(128, n_tok_box, false, false);
    for (int i = 0; i < my_n; ++i) {
      const int b = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      const int t0 = (blockIdx.y + i * gridDim.y) * AT_SB;
      const int ntok = min(AT_SB, Tq - t0);
      const uint32_t tacc = tmem + 256 * b;  // this buffer's four 64-column blocks
      if (lane == 0) {
        // block j = warp of q_lat^T, once its rows of W_uk, the queries and
        // the accumulator buffer (free after the epilogue of sub-block i - 2)
        // are ready
        const int j = warp;
        bool r = ok && (i > 0 || mbar_wait(&sm.full_w[j], 0, AT_WAIT));
        r = r && mbar_wait(&sm.full_q[b], ph, AT_WAIT);
        if (i >= 2) r = r && mbar_wait(&sm.tmem_free[b], ph ^ 1, AT_WAIT);
        if (r) {
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_bf16_ss(tacc + 64 * j, kdesc(sm.w[2 * j + (k >> 2)], (k & 3) * 32),
                        kdesc(sm.q[b][k >> 2], (k & 3) * 32), idesc, k > 0 ? 1u : 0u);
        } else {
          ok = false;
        }
        mma_commit(&sm.mma_done[b]);
      }
      // q_lat^T from TMEM (lane = latent row inside block j, column = token),
      // transposed through shared memory as [token][512]; then every token's
      // 1 KB row goes out in 16-byte stores.
      const bool done = mbar_wait(&sm.mma_done[b], ph, 2 * AT_WAIT);
      tc_fence_after();
      ok = ok && done;
      if (i == my_n - 1) {
        // The CTA's last sub-block (the only one of a decode batch): no MMA
        // reads W_uk any more, so its buffer takes the whole sub-block and
        // one barrier suffices.
        OT* stg = reinterpret_cast<OT*>(sm.w[0]);  // [ntok][512]
        for (int c0 = 0; c0 < ntok; c0 += 16) {
          float v[4][16];
#pragma unroll
          for (int j = 0; j < 4; ++j) tmem_ld16(tacc + lane_base + 64 * j + c0, v[j]);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int dc = 128 * j + 32 * warp + lane;
#pragma unroll
            for (int t = 0; t < 16; ++t)
              stg[(c0 + t) * 512 + dc] = from_f32<OT>(v[j][t] * out_scale);
          }
        }
        named_bar_sync(1, 128);  // the four warps' rows are in place
        if (ok) {
          for (int e = threadIdx.x; e < ntok * 64; e += 128) {
            const int tt = e / 64, u = e % 64;  // 16-byte unit u of token tt's 512 values
            OT* dst = qabs + (static_cast<size_t>(t0 + tt) * s.n_h + h) * R + 8 * u;
            *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(stg + tt * 512 + 8 * u);
          }
        }
        continue;
      }
      for (int c0 = 0; c0 < ntok; c0 += AT_STG_TOK) {
        float v[4][16];
#pragma unroll
        for (int j = 0; j < 4; ++j) tmem_ld16(tacc + lane_base + 64 * j + c0, v[j]);
        tmem_wait_ld();
        if (c0 + AT_STG_TOK >= ntok) {
          // the last TMEM read of this buffer: the MMAs of sub-block i + 2 may
          // overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.tmem_free[b]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int dc = 128 * j + 32 * warp + lane;
#pragma unroll
          for (int t = 0; t < AT_STG_TOK; ++t) sm.stg[t][dc] = from_f32<OT>(v[j][t] * out_scale);
        }
        named_bar_sync(1, 128);  // the four warps' rows are in place
        const int nt = min(AT_STG_TOK, ntok - c0);
        if (ok) {
          for (int e = threadIdx.x; e < nt * 64; e += 128) {
            const int tt = e / 64, u = e % 64;  // 16-byte unit u of token tt's 512 values
            *reinterpret_cast<uint4*>(qabs + (static_cast<size_t>(t0 + c0 + tt) * s.n_h + h) * R +
                                      8 * u) = *reinterpret_cast<const uint4*>(&sm.stg[tt][8 * u]);
          }
        }
        named_bar_sync(1, 128);  // the staging buffer may be refilled
      }
    }
    if (!ok && threadIdx.x == 0) set_error(err, MLA_DEVERR_TIMEOUT);
  } else {
    // rotary block of each query, rotated at the query's own position, from
    // the q_rope box the TMA put in shared memory (128-byte swizzle: dims
    // [8u, 8u + 8) of token row t sit in 16-byte unit u ^ (t & 7)). Lane k
    // owns rotary pair (k, k + 32); warp w4 takes tokens w4, w4 + 4, ...
    // Thread 128 then reloads the buffer with sub-block i + 2.
    const int k = lane, w4 = warp - 4;
    const uint64_t turns = rope_turns[k];
    for (int i = 0; i < my_n; ++i) {
      const int b = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      const int t0 = (blockIdx.y + i * gridDim.y) * AT_SB;
      const int ntok = min(AT_SB, Tq - t0);
      const bool qok = ok && mbar_wait(&sm.full_q[b], ph, AT_WAIT);
      if (!qok) ok = false;
      const uint8_t* qr = sm.q[b][2];
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
      named_bar_sync(2, 128);  // the four warps are done with this buffer's q_rope
      if (threadIdx.x == 128 && i + 2 < my_n) {
        // the MMAs of sub-block i are done with its q_nope
        if (ok && mbar_wait(&sm.mma_done[b], ph, 2 * AT_WAIT)) {
          const int t2 = (blockIdx.y + (i + 2) * gridDim.y) * AT_SB;
          mbar_arrive_expect_tx(&sm.full_q[b], q_tx);
          for (int kc = 0; kc < 3; ++kc)
            tma_load_3d(sm.q[b][kc], &tmap_q, 64 * kc, h, t2, &sm.full_q[b]);
        } else {
          ok = false;
        }
      }
    }
    if (!ok && threadIdx.x == 128) set_error(err, MLA_DEVERR_TIMEOUT);
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
  const int n_tok_box = min(AT_SB, ((Tq + 15) / 16) * 16);
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
  const size_t smem = sizeof(AbsSmem<OT>) + 1024;
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
  // CTAs per head: enough sub-block slices to give every SM a CTA, at most
  // one per sub-block
  static int sms_of[64] = {};
  if (dev >= 0 && dev < 64 && sms_of[dev] == 0 &&
      cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  const int sms = (dev >= 0 && dev < 64) ? sms_of[dev] : 148;
  const int n_sb = (Tq + AT_SB - 1) / AT_SB;
  const int per_head = max(1, min(n_sb, sms / s.n_h));
  cfg.gridDim = dim3(s.n_h, per_head, 1);
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
