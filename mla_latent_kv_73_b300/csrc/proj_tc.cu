// The layer's output projection y = concat_h(o_h) W_o on the tensor cores.
//
// Source: "Multi-head Latent Attention: the KV cache, compressed", section
// "What it costs, said plainly" (W_o, [n_h d_v, d_model], is one of the
// layer's weights; each head's output meets rows [h d_v, (h + 1) d_v)).
//
// y[M x N] = A[M x K] W[K x N], with A the decode outputs (fp32) and W = W_o
// in bf16, row-major (row k holds the N outputs that input k feeds). The
// combine kernel hands A over as a pair of bf16 arrays, hi = bf16(A) and
// lo = bf16(A - hi), which keep about 16 bits of A's mantissa; the tensor
// core multiplies both by W and adds them in its fp32 accumulator.
//
// One CTA per (128 outputs, K slice). It computes the transposed tile
// D[128 x NT] = W^T A^T in TMEM (lane = output, column = token), NT = M
// rounded up to 16 tokens (the MMA's N):
//   - W^T is the MN-major A operand. A TMA box is 64 k-rows of 64 outputs
//     (128 B per row, 128-byte swizzle); the two 64-output halves sit one box
//     apart (the descriptor's leading offset), 8-row groups of k are 1024 B
//     apart (its stride offset), and each K-step of 16 moves 2048 B.
//   - A^T is the K-major B operand: NT token rows of 64 k (128 B), hi and lo
//     in two boxes.
// Warp 4 streams W and A through a 4-stage ring. W is the caller's constant
// weight, so it is requested before the wait for the previous kernel; A is
// requested only after it. Warp 5 issues the 8 MMAs of a stage (hi and lo
// for each of its four K-steps) and frees the stage with a commit. Warps 0-3
// then read the accumulator and store it, coalesced along the outputs, into
// the slice's partial (or straight into y when K is not split). The partials
// are summed in a fixed order by a second kernel, so y does not depend on
// timing.
#include <algorithm>

#include "device_common.cuh"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace mla_ptx;

constexpr int PJ_THREADS = 192;          // warps 0-3 epilogue, 4 producer, 5 MMA issuer
constexpr int PJ_STAGES = 4;
constexpr int PJ_KC = 64;                // k per stage
constexpr uint32_t PJ_WBOX = 64 * 128;   // 64 k-rows x 64 bf16 outputs
constexpr long long PJ_WAIT = 2000000000LL;  // ~1 s

template <int NT>
struct __align__(1024) PjSmem {
  uint8_t w[PJ_STAGES][2][PJ_WBOX];      // [stage][output half]
  uint8_t a[PJ_STAGES][2][NT * 128];     // [stage][hi, lo]: NT token rows x 64 k
  uint64_t full[PJ_STAGES], empty[PJ_STAGES], done;
  uint32_t tmem_base;
};

template <int NT>
__global__ void __launch_bounds__(PJ_THREADS, 1)
proj_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
               int M, int K, int N, int k_split, float* __restrict__ dst, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  PjSmem<NT>& sm = *reinterpret_cast<PjSmem<NT>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                  ~static_cast<uintptr_t>(1023));
  constexpr uint32_t TCOLS = NT <= 32 ? 32 : 64;
  constexpr uint32_t STAGE_TX = 2 * PJ_WBOX + 2 * NT * 128;
  const int n0 = blockIdx.x * 128;
  const int k_begin = blockIdx.y * k_split;
  const int k_end = min(K, k_begin + k_split);
  const int nch = (k_end - k_begin + PJ_KC - 1) / PJ_KC;  // >= 1: the plan leaves no empty slice
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < PJ_STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.done, 1);
    fence_mbarrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&sm.tmem_base, TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 4) {
    if (lane == 0) {
      prefetch_tmap(&tmap_w);
      prefetch_tmap(&tmap_a);
      const int pre = min(nch, PJ_STAGES);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&sm.full[i], STAGE_TX);
        const int k = k_begin + i * PJ_KC;
        tma_load_2d(sm.w[i][0], &tmap_w, n0, k, &sm.full[i]);
        tma_load_2d(sm.w[i][1], &tmap_w, n0 + 64, k, &sm.full[i]);
      }
      griddep_wait();  // A comes from the previous kernel
      for (int i = 0; i < pre; ++i) {
        const int k = k_begin + i * PJ_KC;
        tma_load_3d(sm.a[i][0], &tmap_a, k, 0, 0, &sm.full[i]);
        tma_load_3d(sm.a[i][1], &tmap_a, k, 0, 1, &sm.full[i]);
      }
      int issued = pre;
      bool ok = true;
      for (int i = PJ_STAGES; i < nch; ++i) {
        const int s = i % PJ_STAGES;
        if (!mbar_wait(&sm.empty[s], ((i / PJ_STAGES) - 1) & 1, PJ_WAIT)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&sm.full[s], STAGE_TX);
        const int k = k_begin + i * PJ_KC;
        tma_load_2d(sm.w[s][0], &tmap_w, n0, k, &sm.full[s]);
        tma_load_2d(sm.w[s][1], &tmap_w, n0 + 64, k, &sm.full[s]);
        tma_load_3d(sm.a[s][0], &tmap_a, k, 0, 0, &sm.full[s]);
        tma_load_3d(sm.a[s][1], &tmap_a, k, 0, 1, &sm.full[s]);
        issued = i + 1;
      }
      if (!ok) {
        set_error(err, MLA_DEVERR_TIMEOUT);
        // the loads already issued land before the CTA may exit
        for (int i = max(0, issued - PJ_STAGES); i < issued; ++i)
          mbar_wait(&sm.full[i % PJ_STAGES], (i / PJ_STAGES) & 1, PJ_WAIT);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, NT, true, false);
      bool ok = true;
      for (int i = 0; i < nch; ++i) {
        const int s = i % PJ_STAGES;
        if (!mbar_wait(&sm.full[s], (i / PJ_STAGES) & 1, PJ_WAIT)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < PJ_KC / 16; ++kk) {
          const uint64_t dw = smem_desc(smem_u32(sm.w[s][0]) + 2048u * kk, PJ_WBOX, 1024, kSwizzle128B);
          const uint64_t dh = smem_desc(smem_u32(sm.a[s][0]) + 32u * kk, 16, 1024, kSwizzle128B);
          const uint64_t dl = smem_desc(smem_u32(sm.a[s][1]) + 32u * kk, 16, 1024, kSwizzle128B);
          mma_bf16_ss(tmem, dw, dh, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          mma_bf16_ss(tmem, dw, dl, idesc, 1u);
        }
        mma_commit(&sm.empty[s]);
      }
      if (!ok) set_error(err, MLA_DEVERR_TIMEOUT);
      mma_commit(&sm.done);  // arrives once every MMA issued above is done
    }
  } else {
    // warps 0-3: TMEM lane quarter w holds outputs n0 + 32 w + lane
    griddep_wait();  // the destination is written only after the previous kernel
    const bool ok = mbar_wait(&sm.done, 0, 4 * PJ_WAIT);
    tc_fence_after();
    if (!ok && threadIdx.x == 0) set_error(err, MLA_DEVERR_TIMEOUT);
    const int n = n0 + 32 * warp + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    float* d = dst + static_cast<size_t>(blockIdx.y) * M * N;
#pragma unroll
    for (int c0 = 0; c0 < NT; c0 += 16) {
      float v[16];
      tmem_ld16(tmem + lane_base + c0, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (ok && c0 + i < M && n < N) d[static_cast<size_t>(c0 + i) * N + n] = v[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, TCOLS);
  }
}

template <int NT>
size_t proj_smem() {
  return sizeof(PjSmem<NT>) + 1024;
}

// CTAs of proj_tc_kernel<NT> one SM holds (0 if the kernel cannot be set
// up): its shared memory (with the per-block reservation) against the SM's,
// its TMEM columns against 512. The kernel asks for the largest shared-memory
// carveout, so the launch gets the SM's whole shared memory.
template <int NT>
int proj_resident() {
  static int cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  const int smem = static_cast<int>(proj_smem<NT>());
  int smem_sm = 0, reserved = 0;
  if (cudaFuncSetAttribute(proj_tc_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(proj_tc_kernel<NT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
          cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  constexpr int tcols = NT <= 32 ? 32 : 64;
  int n = smem_sm / (smem + reserved);
  n = std::min(n, std::min(512 / tcols, 2048 / PJ_THREADS));
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

int resident_for(int nt) {
  switch (nt) {
    case 16: return proj_resident<16>();
    case 32: return proj_resident<32>();
    case 48: return proj_resident<48>();
    default: return proj_resident<64>();
  }
}

}  // namespace

bool proj_tc_applies(int M, int K, int N, const void* W) {
  return M >= 1 && M <= PROJ_TC_MAX_TOKENS && K >= 1 && N >= 1 && K % 8 == 0 && N % 8 == 0 &&
         reinterpret_cast<uintptr_t>(W) % 16 == 0;
}

XwPlan proj_tc_plan(int M, int K, int N, int sms) {
  const int nt = ((M + 15) / 16) * 16;
  const int r = resident_for(nt);
  const int tiles = (N + 127) / 128;
  const int chunks = (K + PJ_KC - 1) / PJ_KC;
  int S = r > 0 ? (r * sms) / tiles : 1;
  if (S > chunks) S = chunks;
  if (S > 65535) S = 65535;
  if (S < 1) S = 1;
  const int per = (chunks + S - 1) / S;
  XwPlan p;
  p.k_split = per * PJ_KC;
  p.S = (chunks + per - 1) / per;
  return p;
}

cudaError_t launch_proj_tc(const uint16_t* hilo, int M, int K, const void* W, int N, float* y,
                           float* part, const XwPlan& p, uint32_t* err, cudaStream_t st) {
  if (!proj_tc_applies(M, K, N, W)) return cudaErrorInvalidValue;
  const int nt = ((M + 15) / 16) * 16;
  if (resident_for(nt) < 1) return cudaErrorInvalidConfiguration;
  TmapSpec ws{};
  ws.dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  ws.rank = 2;
  ws.base = W;
  ws.dims[0] = static_cast<uint64_t>(N);
  ws.dims[1] = static_cast<uint64_t>(K);
  ws.strides[0] = static_cast<uint64_t>(N) * 2;
  ws.box[0] = 64;
  ws.box[1] = PJ_KC;
  ws.swizzle = CU_TENSOR_MAP_SWIZZLE_128B;
  TmapSpec as{};
  as.dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  as.rank = 3;
  as.base = hilo;
  as.dims[0] = static_cast<uint64_t>(K);
  as.dims[1] = static_cast<uint64_t>(M);
  as.dims[2] = 2;
  as.strides[0] = static_cast<uint64_t>(K) * 2;
  as.strides[1] = static_cast<uint64_t>(M) * K * 2;
  as.box[0] = PJ_KC;
  as.box[1] = static_cast<uint32_t>(nt);
  as.box[2] = 1;
  as.swizzle = CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap tw, ta;
  if (!get_tmap(ws, &tw) || !get_tmap(as, &ta)) return cudaErrorInvalidValue;
  float* dst = p.S > 1 ? part : y;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((N + 127) / 128, p.S, 1);
  cfg.blockDim = dim3(PJ_THREADS, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  // W streams in while the previous kernel (the combine) finishes
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  switch (nt) {
    case 16:
      cfg.dynamicSmemBytes = proj_smem<16>();
      e = cudaLaunchKernelEx(&cfg, proj_tc_kernel<16>, tw, ta, M, K, N, p.k_split, dst, err);
      break;
    case 32:
      cfg.dynamicSmemBytes = proj_smem<32>();
      e = cudaLaunchKernelEx(&cfg, proj_tc_kernel<32>, tw, ta, M, K, N, p.k_split, dst, err);
      break;
    case 48:
      cfg.dynamicSmemBytes = proj_smem<48>();
      e = cudaLaunchKernelEx(&cfg, proj_tc_kernel<48>, tw, ta, M, K, N, p.k_split, dst, err);
      break;
    default:
      cfg.dynamicSmemBytes = proj_smem<64>();
      e = cudaLaunchKernelEx(&cfg, proj_tc_kernel<64>, tw, ta, M, K, N, p.k_split, dst, err);
      break;
  }
  if (e != cudaSuccess || p.S == 1) return e;
  return launch_sum_splits(part, p.S, static_cast<size_t>(M) * N, y, st);
}

}  // namespace mla
