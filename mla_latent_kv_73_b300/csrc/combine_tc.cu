// a4 + a5 (tensor-core variant): merge the split-KV partials by their
// log-sum-exps, then up-project the latent output through W_uv.
//
//   lse   = log sum_s exp(lse_s)
//   o_lat = sum_s exp(lse_s - lse) * o_s          (each o_s already divided by l_s)
//   out   = W_uv[h] o_lat                          (d_v = 128 outputs per head)
//
// The value up-projection runs once per head and query, after the weighted
// sum, rather than once per cached token. Source: "Multi-head Latent
// Attention and KV Cache Compression", section "The absorption trick and
// decoupled RoPE" (W_uv is absorbed on the output side the way W_uk is on the
// query side).
//
// One CTA per (head, up to 32 query tokens). At entry, one thread starts the
// TMA of the head's whole W_uv slice (128 KB, eight 128 x 64 boxes) so the
// weight stream overlaps the combine. All threads then merge the partials of
// their tokens into o_lat (fp32 in registers), split each value into a bf16
// high part and a bf16 remainder, and store both as MMA operands in shared
// memory. Four threads issue the product out^T = W_uv[h] (o_hi + o_lo)^T, each
// 2 x 8 MMAs with M = 128 outputs, N = tokens over a quarter of K = 512 into
// its own TMEM accumulator. The hi + lo split keeps about 16 bits of o_lat's
// mantissa, so rounding o_lat for the tensor core costs no measurable
// accuracy. Four warps read the four fp32 accumulators from TMEM, one output
// column per lane, add them in a fixed order and store the sum. For the
// layer step they also store the sum as a bf16 hi + lo pair, the operand of
// the tensor-core W_o projection.
//
// The latent mode (mla_decode_latent, the attention core alone) keeps only
// the merge: each thread writes its 8 merged o_lat values straight to
// global memory, with no W_uv, TMEM or MMA.
#include <cmath>
#include <cstring>

#include "device_common.cuh"
#include "plan.cuh"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace mla_ptx;

constexpr int CT_TOK = 32;                   // query tokens per CTA (MMA N)
constexpr int CT_THREADS = 256;
constexpr uint32_t CT_WBOX = 128 * 128;      // 128 rows x 64 bf16
constexpr uint32_t CT_OBOX = CT_TOK * 128;   // 32 token rows x 64 bf16
constexpr long long CT_WAIT = 2000000000LL;

// Per token of the CTA: the first and last range holding its pieces, and its
// row offset inside a slot of the partials.
struct CombPlan {
  int c_lo[CT_TOK], c_hi[CT_TOK], row_off[CT_TOK];
};

struct __align__(1024) CombSmem {
  uint8_t w[8][CT_WBOX];          // K-chunk kc of W_uv[h]: 128 output rows x 64 latent dims
  uint8_t o[2][8][CT_OBOX];       // [hi/lo][K-chunk]: token rows x 64 latent dims
  uint64_t wfull, done;
  uint32_t tmem_base;
  CombPlan plan;
};

// Shared memory before the range starts and merge weights: the whole
// CombSmem, or only the plan in the latent mode.
template <bool LATENT>
constexpr size_t comb_head_bytes() {
  return LATENT ? (sizeof(CombPlan) + 15) / 16 * 16 : sizeof(CombSmem);
}

__device__ __forceinline__ uint64_t kdesc(const void* base, uint32_t byte_off) {
  return smem_desc(smem_u32(base) + byte_off, 16, 1024, kSwizzle128B);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// LATENT: merge only, writing o_lat [B*n_q][n_h][512] fp32 to `out` (no W_uv,
// no TMEM, no MMA); the attention core alone (mla_decode_latent).
template <bool LATENT>
__global__ void __launch_bounds__(CT_THREADS, 1)
combine_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, int n_h,
                  const int32_t* __restrict__ tiles, const int32_t* __restrict__ prefix,
                  const long long* __restrict__ bounds, int B, int n_q, Partition p,
                  const float* __restrict__ part_o,
                  const float* __restrict__ part_lse, float* __restrict__ out,
                  uint16_t* __restrict__ hilo, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  CombSmem& sm = *reinterpret_cast<CombSmem*>(base);  // touched only outside the latent mode
  CombPlan& pl = LATENT ? *reinterpret_cast<CombPlan*>(base) : sm.plan;
  long long* rb = reinterpret_cast<long long*>(base + comb_head_bytes<LATENT>());  // [C + 1] range starts
  const int h = blockIdx.x, t0 = blockIdx.y * CT_TOK;
  const int Tq = B * n_q, ntok = min(CT_TOK, Tq - t0);
  const int n_box = ((ntok + 15) / 16) * 16;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  uint32_t tmem = 0;
  if constexpr (!LATENT) {
    if (threadIdx.x == 0) {
      mbar_init(&sm.wfull, 1);
      mbar_init(&sm.done, 4);  // one commit per K quarter
      fence_mbarrier_init();
    }
    if (warp == 1) {
      tmem_alloc(&sm.tmem_base, 128);
      tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tmem = sm.tmem_base;
    // With programmatic dependent launch this CTA may start while the
    // attention kernel still runs. The packed W_uv is complete and never
    // written once its handle exists, so its loads start at once; everything
    // the attention kernel writes is read only after the wait.
    if (threadIdx.x == 0) {
      prefetch_tmap(&tmap_w);
      mbar_arrive_expect_tx(&sm.wfull, 8 * CT_WBOX);
      for (int kc = 0; kc < 8; ++kc) tma_load_2d(sm.w[kc], &tmap_w, 64 * kc, h * 128, &sm.wfull);
    }
  }
  griddep_wait();
  // the next kernel (its weights are constant) may start its prologue now;
  // it waits for this one to finish before it reads anything this one writes
  griddep_launch_dependents();

  // 1. per token: the CTAs holding its pieces and their merge weights
  //    exp(lse_s - lse). The plan loads of all tokens go out together (the
  //    range starts, and each token's tiles and prefix in one round trip);
  //    then half a warp per token, its lanes taking the pieces, loads the
  //    lse values, so two tokens per warp cost one more round trip.
  const long long T_all = prefix[B];
  for (int c = threadIdx.x; c <= p.C; c += CT_THREADS) rb[c] = bounds[c];  // all 0 without tiles
  int my_tiles = 0, my_off = 0;
  long long my_first = 0;
  if (threadIdx.x < ntok) {
    const int tok = t0 + threadIdx.x, b = tok / n_q, qi = tok % n_q;
    const int r = qi * n_h + h, g = r / p.RG, rr = r % p.RG;
    my_off = (g * B + b) * p.RG + rr;  // row of slot (c + g*B + b) is c*RG + off
    my_tiles = tiles[b];
    my_first = static_cast<long long>(g) * T_all + prefix[b];
  }
  __syncthreads();  // range starts in place
  if (threadIdx.x < CT_TOK) {
    int c0 = 0, c1 = -1;
    if (my_tiles > 0) {
      c0 = range_of_item(rb, p.C, my_first);
      c1 = range_of_item(rb, p.C, my_first + my_tiles - 1);
    }
    pl.c_lo[threadIdx.x] = c0;
    pl.c_hi[threadIdx.x] = c1;
    pl.row_off[threadIdx.x] = my_off;
  }
  __syncthreads();
  float* wts = reinterpret_cast<float*>(rb + p.C + 1);  // [CT_TOK][C + 1] merge weights
  for (int tb = 0; tb < ntok; tb += 2 * (CT_THREADS / 32)) {
    const int t = tb + 2 * warp + (lane >> 4), hl = lane & 15;
    const bool live = t < ntok;
    const int c0 = live ? pl.c_lo[t] : 0, c1 = live ? pl.c_hi[t] : -1;
    const int off = live ? pl.row_off[t] : 0;
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
    if (live && hl == 0 && M == -INFINITY) pl.c_hi[t] = -1;  // no piece holds a visible token
  }
  __syncthreads();

  // 2. o_lat = weighted sum of the partials; a thread owns 8 latent dims of
  // tokens g, g + 4, g + 8, ... (g = thread / 64) and keeps the loads of four
  // of its tokens, four pieces each, in flight together.
  {
    const int u = threadIdx.x % 64;  // 16-byte unit: latent dims [8u, 8u + 8)
    const int kc = u / 8, uu = u % 8;
    const int g = threadIdx.x / 64;
    for (int tb = 0; tb < CT_TOK; tb += 16) {
      float acc[4][8];
      int lo[4], hi[4];
      size_t off[4];
      int nb = 0;  // batches of four pieces
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j][i] = 0.f;
        const int tt = tb + g + 4 * j;
        lo[j] = 0;
        hi[j] = -1;
        off[j] = 0;
        if (tt < ntok) {
          lo[j] = pl.c_lo[tt];
          hi[j] = pl.c_hi[tt];
          off[j] = pl.row_off[tt];
          nb = max(nb, (hi[j] - lo[j] + 4) / 4);
        }
      }
      for (int bb = 0; bb < nb; ++bb) {
        float4 va[4][4], vb[4][4];
        float wg[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float* w = wts + (tb + g + 4 * j) * (p.C + 1) - lo[j];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = lo[j] + 4 * bb + q;
            const bool in = c <= hi[j];
            const int cj = in ? c : max(lo[j], 0);
            wg[j][q] = in ? w[c] : 0.f;  // empty ranges carry weight 0
            const float4* src = reinterpret_cast<const float4*>(
                part_o + (static_cast<size_t>(cj) * p.RG + off[j]) * 512 + 8 * u);
            va[j][q] = in ? src[0] : make_float4(0.f, 0.f, 0.f, 0.f);
            vb[j][q] = in ? src[1] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (wg[j][q] == 0.f) continue;  // also skips partials no range wrote
            acc[j][0] = fmaf(wg[j][q], va[j][q].x, acc[j][0]);
            acc[j][1] = fmaf(wg[j][q], va[j][q].y, acc[j][1]);
            acc[j][2] = fmaf(wg[j][q], va[j][q].z, acc[j][2]);
            acc[j][3] = fmaf(wg[j][q], va[j][q].w, acc[j][3]);
            acc[j][4] = fmaf(wg[j][q], vb[j][q].x, acc[j][4]);
            acc[j][5] = fmaf(wg[j][q], vb[j][q].y, acc[j][5]);
            acc[j][6] = fmaf(wg[j][q], vb[j][q].z, acc[j][6]);
            acc[j][7] = fmaf(wg[j][q], vb[j][q].w, acc[j][7]);
          }
      }
      if constexpr (LATENT) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int tt = tb + g + 4 * j;
          if (tt >= ntok) continue;
          float4* dst = reinterpret_cast<float4*>(
              out + (static_cast<size_t>(t0 + tt) * n_h + h) * 512 + 8 * u);
          dst[0] = make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
          dst[1] = make_float4(acc[j][4], acc[j][5], acc[j][6], acc[j][7]);
        }
        continue;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tt = tb + g + 4 * j;
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat162 hv = __floats2bfloat162_rn(acc[j][2 * i], acc[j][2 * i + 1]);
          hw[i] = *reinterpret_cast<const uint32_t*>(&hv);
          lw[i] = pack_bf16x2(acc[j][2 * i] - __low2float(hv), acc[j][2 * i + 1] - __high2float(hv));
        }
        const uint32_t o = tt * 128 + ((uu ^ (tt & 7)) * 16);
        *reinterpret_cast<uint4*>(sm.o[0][kc] + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(sm.o[1][kc] + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    }
  }
  if constexpr (LATENT) return;
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // 3. out^T = W_uv[h] o_lat^T on the tensor core: K quarter i = warp i
  // (K-steps 8i .. 8i + 7, both parts) into accumulator columns [32i, 32i + 32)
  if (warp < 4 && lane == 0) {
    if (mbar_wait(&sm.wfull, 0, CT_WAIT)) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, n_box, false, false);
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int k = 8 * warp + kk;
          mma_bf16_ss(tmem + 32 * warp, kdesc(sm.w[k >> 2], (k & 3) * 32),
                      kdesc(sm.o[part][k >> 2], (k & 3) * 32), idesc,
                      (part == 0 && kk == 0) ? 0u : 1u);
        }
    } else {
      set_error(err, MLA_DEVERR_TIMEOUT);
    }
    mma_commit(&sm.done);
  }
  if (warp < 4) {
    // out^T from TMEM (lane = output dim, column = token), transposed
    // through the o_lat staging (the MMAs are done with it) as
    // [token][128] fp32, then each token's 512-byte row goes out in 16-byte
    // stores.
    const bool done = mbar_wait(&sm.done, 0, 2 * CT_WAIT);
    tc_fence_after();
    float* stg = reinterpret_cast<float*>(sm.o[0][0]);  // [n_box][128]
    if (done) {
      const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
      const int dv = 32 * warp + lane;
      for (int c0 = 0; c0 < n_box; c0 += 16) {
        float v[16], v1[16], v2[16], v3[16];
        tmem_ld16(tmem + lane_base + c0, v);
        tmem_ld16(tmem + lane_base + 32 + c0, v1);
        tmem_ld16(tmem + lane_base + 64 + c0, v2);
        tmem_ld16(tmem + lane_base + 96 + c0, v3);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) stg[(c0 + i) * 128 + dv] = (v[i] + v1[i]) + (v2[i] + v3[i]);
      }
    } else if (warp == 0 && lane == 0) {
      set_error(err, MLA_DEVERR_TIMEOUT);
    }
    named_bar_sync(1, 128);  // the four warps' columns are in place
    if (done) {
      const size_t plane = static_cast<size_t>(Tq) * n_h * 128;  // elements of hi (and of lo)
      for (int i = threadIdx.x; i < ntok * 32; i += 128) {
        const int tt = i / 32, u = i % 32;  // 16-byte unit u of token tt's 128 outputs
        const size_t e = (static_cast<size_t>(t0 + tt) * n_h + h) * 128 + 4 * u;
        const float4 v = *reinterpret_cast<const float4*>(stg + tt * 128 + 4 * u);
        *reinterpret_cast<float4*>(out + e) = v;
        if (hilo) {
          const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y);
          const __nv_bfloat162 h1 = __floats2bfloat162_rn(v.z, v.w);
          *reinterpret_cast<uint2*>(hilo + e) =
              make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
          *reinterpret_cast<uint2*>(hilo + plane + e) =
              make_uint2(pack_bf16x2(v.x - __low2float(h0), v.y - __high2float(h0)),
                         pack_bf16x2(v.z - __low2float(h1), v.w - __high2float(h1)));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

}  // namespace

bool combine_tc_supported(const Shape& s, mla_dtype dt) {
  return dt == MLA_BF16 && s.d_c == 512 && s.d_v == 128;
}

namespace {

template <bool LATENT>
cudaError_t combine_tc_t(const Shape& s, const CUtensorMap& tw, int B, int n_q,
                         const Partition& p, const WsView& ws, float* out, uint16_t* hilo,
                         uint32_t* err, cudaStream_t st) {
  const int Tq = B * n_q;
  const size_t smem = comb_head_bytes<LATENT>() + 1024 + sizeof(long long) * (p.C + 1) +
                      sizeof(float) * CT_TOK * (p.C + 1);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  static int attr_bytes[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || attr_bytes[dev] < static_cast<int>(smem)) {
    cudaError_t e = cudaFuncSetAttribute(combine_tc_kernel<LATENT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_bytes[dev] = static_cast<int>(smem);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.n_h, (Tq + CT_TOK - 1) / CT_TOK, 1);
  cfg.blockDim = dim3(CT_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // may start while the attention kernel finishes (see the kernel's wait)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_tc_kernel<LATENT>, tw, s.n_h,
                            static_cast<const int32_t*>(ws.tiles),
                            static_cast<const int32_t*>(ws.prefix),
                            static_cast<const long long*>(ws.bounds), B, n_q, p,
                            static_cast<const float*>(ws.part_o),
                            static_cast<const float*>(ws.part_lse), out, hilo, err);
}

}  // namespace

cudaError_t launch_combine_tc(const Shape& s, const Weights* w, int B, int n_q,
                              const Partition& p, const WsView& ws, float* out, uint16_t* hilo,
                              uint32_t* err, cudaStream_t st) {
  TmapSpec spec{};
  spec.dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  spec.rank = 2;
  spec.base = w->w_uv;
  spec.dims[0] = 512;
  spec.dims[1] = static_cast<uint64_t>(s.n_h) * 128;
  spec.strides[0] = 1024;
  spec.box[0] = 64;
  spec.box[1] = 128;
  spec.swizzle = CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap tw;
  if (!get_tmap(spec, &tw)) return cudaErrorInvalidValue;
  return combine_tc_t<false>(s, tw, B, n_q, p, ws, out, hilo, err, st);
}

bool combine_latent_tc_supported(const Shape& s) { return s.d_c == 512; }

cudaError_t launch_combine_latent_tc(const Shape& s, int B, int n_q, const Partition& p,
                                     const WsView& ws, float* olat, uint32_t* err,
                                     cudaStream_t st) {
  CUtensorMap unused;
  std::memset(&unused, 0, sizeof(unused));
  return combine_tc_t<true>(s, unused, B, n_q, p, ws, olat, nullptr, err, st);
}

}  // namespace mla
