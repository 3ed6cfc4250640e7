// a3 (tensor-core variant): split-KV attention of absorbed queries over the
// paged latent cache on tcgen05 / TMEM, with TMA-staged tiles.
//
//   S     = Q K^T * scale        Q: [64 query rows x 576], K: [64 tokens x 576]
//   P     = online softmax of S (causal mask j <= pos_q), bf16
//   O^T  += C^T P^T              C: the 512 latent columns of the same tile
//
// Sources: "Multi-head Latent Attention: the KV cache, compressed", sections
// "Absorption: the part that makes it free" (queries are projected into
// latent space and dotted against the cache; keys are never built) and
// "RoPE, and why the explanations stop here" (the score is the sum of a
// content part and a decoupled RoPE part, which a single 576-wide dot
// product over [c | k_rope] computes); "Multi-head Latent Attention and KV
// Cache Compression", section "The absorption trick and decoupled RoPE"
// (the output is the softmax-weighted sum of latents, up-projected later).
//
// Why this shape on sm_103a. All heads share one 576-wide key row and one
// 512-wide value row per token, so both products are dense contractions.
// The fp32 latent accumulator of 64 query rows is 64 x 512 x 4 B = 128 KB.
// Kept transposed (latent dims in TMEM lanes, query rows in columns), it
// fills 4 M=128 blocks of 64 columns = 256 of the 512 TMEM columns. That
// leaves room for two 64-column score buffers, so the score MMA of tile i+1
// overlaps the softmax of tile i. The score MMA uses M = 64 query rows.
// The value MMA reads its A operand (C^T) straight from the same swizzled
// tile in shared memory, as an MN-major operand, so the tile is loaded once
// and feeds both products.
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: Q rows once per piece, then 9 boxes of 64 x 64
//               bf16 per 64-token page, 2-stage ring
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2..5  softmax (query row r lives in TMEM lane 32*(r/16) + r%16),
//               lazy rescale of O^T, and the epilogue of each piece
//
// Lazy rescale: a row's running max is only raised when the new max exceeds
// it by more than 8 (log2 units). Otherwise P is computed against the stale
// max, so its entries stay <= 2^8. The final division by the row sum l
// cancels the offset exactly.
//
// Every mbarrier wait is bounded. On a timeout the CTA sets
// MLA_DEVERR_TIMEOUT, stops issuing work, drains what it issued, frees
// TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "device_common.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace {

using namespace mla_ptx;

constexpr int TC_ROWS = 64;                 // query rows per group (score MMA M)
constexpr int TC_TOK = 64;                  // tokens per tile = page size
constexpr int TC_KCH = 9;                   // 576 / 64 column chunks
constexpr int TC_STAGES = 2;
constexpr int TC_THREADS = 192;
constexpr uint32_t CHUNK_BYTES = 64 * 128;  // 64 rows x 128 B (one 128B-swizzled box)
constexpr uint32_t TILE_BYTES = TC_KCH * CHUNK_BYTES;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;                // two score buffers at columns 0 and 64
constexpr uint32_t TM_O = 128;              // O^T block j at columns 128 + 64 j
constexpr long long WAIT_LIMIT = 4000000000LL;  // ~2 s at 2 GHz
constexpr float RESCALE_THRESHOLD = 8.f;        // log2 units

struct __align__(1024) TcSmem {
  uint8_t q[TC_KCH][CHUNK_BYTES];
  uint8_t kv[TC_STAGES][TC_KCH][CHUNK_BYTES];
  uint8_t p[CHUNK_BYTES];  // 64 rows x 64 tokens bf16, K-major, 128B swizzle
  uint64_t kv_full[TC_STAGES], kv_empty[TC_STAGES];
  uint64_t q_full, q_empty;
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full, p_empty;
  uint64_t o_full, o_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  float row_alpha[TC_ROWS];
  float row_inv_l[TC_ROWS];
};

struct TcArgs {
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* tiles;
  const int32_t* prefix;
  float* part_o;
  float* part_lse;
  uint32_t* err;
  int num_blocks, max_blocks, B, n_q, n_h, RG, G, C;
  float scale_log2;
};

// One piece: consecutive tiles of one (group, sequence) inside a CTA's range.
struct Piece {
  int g, b, t_first, n_tiles;
};

__device__ __forceinline__ Piece locate_piece(long long it, long long end, long long T_all,
                                              const int32_t* prefix, const int32_t* tiles,
                                              int B) {
  Piece pc;
  pc.g = static_cast<int>(it / T_all);
  const long long rem = it % T_all;
  int lo = 0, hi = B;  // largest b with prefix[b] <= rem
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= rem) lo = mid; else hi = mid;
  }
  pc.b = lo;
  pc.t_first = static_cast<int>(rem - prefix[lo]);
  const long long stop = min(end, static_cast<long long>(pc.g) * T_all + prefix[lo] + tiles[lo]);
  pc.n_tiles = static_cast<int>(stop - it);
  return pc;
}

__device__ __forceinline__ void note_timeout(TcSmem& sm, uint32_t* err) {
  *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
  set_error(err, MLA_DEVERR_TIMEOUT);
}

// Descriptors. Q and K tiles: K-major, 128 B rows, 8-row groups 1024 B apart.
// Advancing K by 16 bf16 (32 B) inside a swizzle atom advances the start address.
__device__ __forceinline__ uint64_t desc_kmajor(const void* chunk, uint32_t k_byte_off) {
  return smem_desc(smem_u32(chunk) + k_byte_off, 16, 1024, kSwizzle128B);
}
// C^T as an MN-major operand: latent dims are contiguous (64 per 128 B row, next
// 64 dims one box = 8192 B further), tokens step 128 B, 8-token groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_ct(const void* chunk, uint32_t token_byte_off) {
  return smem_desc(smem_u32(chunk) + token_byte_off, CHUNK_BYTES, 1024, kSwizzle128B);
}

__global__ void __launch_bounds__(TC_THREADS, 1)
attend_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                 const __grid_constant__ CUtensorMap tmap_kv, TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem& sm = *reinterpret_cast<TcSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const long long T_all = a.prefix[a.B];
  const long long N = T_all * a.G;
  if (N == 0) return;
  const long long it_begin = range_begin(blockIdx.x, N, a.C);
  const long long it_end = range_begin(blockIdx.x + 1, N, a.C);
  if (it_begin == it_end) return;
  const int rows_total = a.n_q * a.n_h;

  if (threadIdx.x == 0) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_empty[i], 4);
    }
    mbar_init(&sm.p_full, 1);
    mbar_init(&sm.p_empty, 1);
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.o_empty, 1);
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmap_q);
      prefetch_tmap(&tmap_kv);
      const uint64_t pol = policy_evict_first();
      uint32_t kv_it = 0;
      int piece_idx = 0;
      uint32_t issued[TC_STAGES] = {0, 0};  // loads issued per stage
      for (long long it = it_begin; it < it_end && !*reinterpret_cast<volatile int*>(&sm.abort_flag);) {
        const Piece pc = locate_piece(it, it_end, T_all, a.prefix, a.tiles, a.B);
        if (piece_idx > 0 && !mbar_wait(&sm.q_empty, (piece_idx - 1) & 1, WAIT_LIMIT)) {
          note_timeout(sm, a.err);
          break;
        }
        mbar_arrive_expect_tx(&sm.q_full, TILE_BYTES);
        const int qrow0 = pc.b * rows_total + pc.g * a.RG;
        for (int c = 0; c < TC_KCH; ++c) tma_load_2d(sm.q[c], &tmap_q, 64 * c, qrow0, &sm.q_full);
        for (int t = pc.t_first; t < pc.t_first + pc.n_tiles; ++t) {
          const int s = kv_it % TC_STAGES;
          const uint32_t n = kv_it / TC_STAGES;
          if (kv_it >= TC_STAGES && !mbar_wait(&sm.kv_empty[s], (n - 1) & 1, WAIT_LIMIT)) {
            note_timeout(sm, a.err);
            break;
          }
          int page = a.page_table[static_cast<size_t>(pc.b) * a.max_blocks + t];
          if (page < 0 || page >= a.num_blocks) {
            set_error(a.err, MLA_DEVERR_PAGE_RANGE);
            page = 0;
          }
          mbar_arrive_expect_tx(&sm.kv_full[s], TILE_BYTES);
          for (int c = 0; c < TC_KCH; ++c)
            tma_load_2d_hint(sm.kv[s][c], &tmap_kv, 64 * c, page * TC_TOK, &sm.kv_full[s], pol);
          ++issued[s];
          ++kv_it;
        }
        ++piece_idx;
        it += pc.n_tiles;
      }
      // Never leave a TMA write in flight past the end of the CTA.
      for (int s = 0; s < TC_STAGES; ++s)
        if (issued[s] > 0) mbar_wait(&sm.kv_full[s], (issued[s] - 1) & 1, WAIT_LIMIT);
      if (piece_idx > 0) mbar_wait(&sm.q_full, (piece_idx - 1) & 1, WAIT_LIMIT);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(TC_ROWS, TC_TOK, false, false);
      const uint32_t idPV = idesc_bf16_f32(128, a.RG, true, false);
      uint32_t kv_it = 0;
      int piece_idx = 0;
      bool pend = false, pend_first = false, pend_last = false;
      uint32_t pend_it = 0;
      int pend_piece = 0;
      bool ok = true;

      auto issue_pv = [&](uint32_t pit, bool first, bool last, int ppiece) -> bool {
        if (!mbar_wait(&sm.p_full, pit & 1, WAIT_LIMIT)) return false;
        if (first && ppiece > 0 && !mbar_wait(&sm.o_empty, (ppiece - 1) & 1, WAIT_LIMIT))
          return false;
        tc_fence_after();
        const int s = pit % TC_STAGES;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = desc_ct(sm.kv[s][2 * j], kk * 2048);
            const uint64_t bd = desc_kmajor(sm.p, kk * 32);
            mma_bf16_ss(tmem + TM_O + 64 * j, ad, bd, idPV, (first && kk == 0) ? 0u : 1u);
          }
        }
        mma_commit(&sm.kv_empty[s]);
        mma_commit(&sm.p_empty);
        if (last) mma_commit(&sm.o_full);
        return true;
      };

      for (long long it = it_begin; it < it_end && ok;) {
        const Piece pc = locate_piece(it, it_end, T_all, a.prefix, a.tiles, a.B);
        if (!mbar_wait(&sm.q_full, piece_idx & 1, WAIT_LIMIT)) { ok = false; break; }
        tc_fence_after();
        for (int i = 0; i < pc.n_tiles; ++i) {
          const int sb = kv_it & 1;
          if (kv_it >= 2 && !mbar_wait(&sm.s_empty[sb], ((kv_it >> 1) - 1) & 1, WAIT_LIMIT)) {
            ok = false;
            break;
          }
          const int s = kv_it % TC_STAGES;
          if (!mbar_wait(&sm.kv_full[s], (kv_it / TC_STAGES) & 1, WAIT_LIMIT)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4 * TC_KCH; ++k) {
            const int c = k >> 2;
            const uint32_t off = (k & 3) * 32;
            mma_bf16_ss(tmem + TM_S + 64 * sb, desc_kmajor(sm.q[c], off),
                        desc_kmajor(sm.kv[s][c], off), idS, k > 0 ? 1u : 0u);
          }
          mma_commit(&sm.s_full[sb]);
          if (i == pc.n_tiles - 1) mma_commit(&sm.q_empty);
          if (pend && !issue_pv(pend_it, pend_first, pend_last, pend_piece)) {
            ok = false;
            break;
          }
          pend = true;
          pend_it = kv_it;
          pend_first = (i == 0);
          pend_last = (i == pc.n_tiles - 1);
          pend_piece = piece_idx;
          ++kv_it;
        }
        ++piece_idx;
        it += pc.n_tiles;
      }
      if (ok && pend && !issue_pv(pend_it, pend_first, pend_last, pend_piece)) ok = false;
      if (!ok) note_timeout(sm, a.err);
      // Wait until every MMA issued above has completed before TMEM is freed.
      mma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, WAIT_LIMIT);
    }
  } else {
    // ------------------------------------------------------------ softmax warps 2..5
    const int qd = warp & 3;                 // TMEM lane quarter this warp may access
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    const int row = 16 * qd + lane;          // score row held by this lane (lane < 16)
    const bool lane_has_row = lane < 16;
    const int tid_sm = threadIdx.x - 64;     // 0..127
    uint32_t kv_it = 0;
    int piece_idx = 0;
    bool ok = true;
    for (long long it = it_begin; it < it_end && ok;) {
      const Piece pc = locate_piece(it, it_end, T_all, a.prefix, a.tiles, a.B);
      const int L = a.seq_lens[pc.b];
      const int rg = pc.g * a.RG + row;
      const int rows_valid = min(a.RG, rows_total - pc.g * a.RG);
      const bool row_ok = lane_has_row && row < rows_valid;
      const int pos_q = L - a.n_q + (row_ok ? rg / a.n_h : 0);
      float m = -INFINITY, l = 0.f;

      for (int i = 0; i < pc.n_tiles; ++i) {
        const int t = pc.t_first + i;
        const int sb = kv_it & 1;
        const int s = kv_it % TC_STAGES;
        bool w_ok = mbar_wait(&sm.s_full[sb], (kv_it >> 1) & 1, WAIT_LIMIT);
        if (named_bar_or(1, 128, !w_ok)) { ok = false; break; }
        tc_fence_after();
        float sc[TC_TOK];
#pragma unroll
        for (int c0 = 0; c0 < TC_TOK; c0 += 16) {
          float v[16];
          tmem_ld16(tmem + lane_base + TM_S + 64 * sb + c0, v);
#pragma unroll
          for (int k = 0; k < 16; ++k) sc[c0 + k] = v[k];
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.s_empty[sb]);

        const int j0 = t * TC_TOK;
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < TC_TOK; ++c) {
          const bool valid = row_ok && (j0 + c <= pos_q);
          sc[c] = valid ? sc[c] * a.scale_log2 : -INFINITY;
          mx = fmaxf(mx, sc[c]);
        }
        const float m_new = fmaxf(m, mx);
        const bool first = (i == 0);
        const bool need = !first && (m_new > m + RESCALE_THRESHOLD);
        const float m_use = (first || need) ? m_new : m;
        const float alpha = (m == -INFINITY || first) ? 0.f : exp2f(m - m_use);

        // P buffer free and O^T stable once the previous value MMA has finished.
        w_ok = (kv_it == 0) || mbar_wait(&sm.p_empty, (kv_it - 1) & 1, WAIT_LIMIT);
        if (named_bar_or(1, 128, !w_ok)) { ok = false; break; }
        tc_fence_after();
        const bool any = named_bar_or(1, 128, need && row_ok);
        if (any) {
          if (lane_has_row) sm.row_alpha[row] = need && row_ok ? alpha : 1.f;
          named_bar_sync(1, 128);
          for (int j = 0; j < 4; ++j) {
            for (int c0 = 0; c0 < a.RG; c0 += 16) {
              float v[16];
              const uint32_t ta = tmem + lane_base + TM_O + 64 * j + c0;
              tmem_ld16(ta, v);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 16; ++k) v[k] *= sm.row_alpha[c0 + k];
              tmem_st16(ta, v);
            }
          }
          tmem_wait_st();
        }
        // P row -> shared memory (bf16, 128B-swizzled K-major), row sums
        if (lane_has_row) {
          float psum = 0.f;
          uint8_t* prow = sm.p + row * 128;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float x0 = sc[ch * 8 + 2 * k], x1 = sc[ch * 8 + 2 * k + 1];
              const float p0 = (x0 == -INFINITY) ? 0.f : exp2f(x0 - m_use);
              const float p1 = (x1 == -INFINITY) ? 0.f : exp2f(x1 - m_use);
              const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
              psum += __low2float(pb) + __high2float(pb);
              w[k] = *reinterpret_cast<const uint32_t*>(&pb);
            }
            *reinterpret_cast<uint4*>(prow + ((ch ^ (row & 7)) * 16)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (row_ok) {
            l = l * alpha + psum;
            m = m_use;
          }
        }
        // Rows past the end of the sequence may hold anything; zero their
        // latent columns so that 0 * garbage cannot reach the accumulator.
        if (j0 + TC_TOK > L) {
          const int r0 = L - j0;  // first invalid row in this tile
          const int nrow = TC_TOK - r0;
          for (int i2 = tid_sm; i2 < nrow * 8 * 8; i2 += 128) {
            const int rr = r0 + i2 / 64, ch = (i2 / 8) % 8, u = i2 % 8;
            *reinterpret_cast<uint4*>(sm.kv[s][ch] + rr * 128 + u * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(1, 128);
        if (tid_sm == 0) mbar_arrive(&sm.p_full);
        ++kv_it;
      }
      if (!ok) break;

      // ---- epilogue of the piece: O^T / l -> workspace slot
      const bool w_ok = mbar_wait(&sm.o_full, piece_idx & 1, WAIT_LIMIT);
      if (named_bar_or(1, 128, !w_ok)) { ok = false; break; }
      tc_fence_after();
      const int slot = blockIdx.x + pc.g * a.B + pc.b;
      if (lane_has_row) {
        sm.row_inv_l[row] = (row_ok && l > 0.f) ? 1.f / l : 0.f;
        if (row_ok)
          a.part_lse[static_cast<size_t>(slot) * a.RG + row] =
              l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
      named_bar_sync(1, 128);
      float* dst = a.part_o + static_cast<size_t>(slot) * a.RG * 512;
      for (int j = 0; j < 4; ++j) {
        for (int c0 = 0; c0 < a.RG; c0 += 16) {
          float v[16];
          tmem_ld16(tmem + lane_base + TM_O + 64 * j + c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int n = c0 + k;
            if (n < rows_valid) dst[static_cast<size_t>(n) * 512 + 128 * j + 32 * qd + lane] =
                v[k] * sm.row_inv_l[n];
          }
        }
      }
      tc_fence_before();
      named_bar_sync(1, 128);
      if (tid_sm == 0) mbar_arrive(&sm.o_empty);
      ++piece_idx;
      it += pc.n_tiles;
    }
    if (!ok && tid_sm == 0) note_timeout(sm, a.err);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_rows_map(CUtensorMap* m, const void* base, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {576, rows};
  cuuint64_t strides[1] = {576 * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool attend_tc_supported(const Shape& s, mla_dtype dt) {
  return dt == MLA_BF16 && s.d_c == 512 && s.d_r == 64 && s.bs == TC_TOK;
}

size_t attend_tc_smem_bytes() { return sizeof(TcSmem) + 1024; }

cudaError_t launch_attend_tc(const Shape& s, const void* cache, int num_blocks,
                             const int32_t* page_table, int max_blocks, int B, int n_q,
                             const Partition& p, const WsView& ws, const int32_t* seq_lens,
                             uint32_t* err, cudaStream_t st) {
  CUtensorMap tq, tkv;
  const uint64_t q_rows = static_cast<uint64_t>(B) * n_q * s.n_h;
  if (!make_rows_map(&tq, ws.qabs, q_rows)) return cudaErrorInvalidValue;
  if (!make_rows_map(&tkv, cache, static_cast<uint64_t>(num_blocks) * TC_TOK))
    return cudaErrorInvalidValue;
  TcArgs a;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.tiles = ws.tiles;
  a.prefix = ws.prefix;
  a.part_o = ws.part_o;
  a.part_lse = ws.part_lse;
  a.err = err;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks;
  a.B = B;
  a.n_q = n_q;
  a.n_h = s.n_h;
  a.RG = p.RG;
  a.G = p.G;
  a.C = p.C;
  a.scale_log2 = s.scale * 1.4426950408889634f;
  const size_t smem = attend_tc_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  attend_tc_kernel<<<p.C, TC_THREADS, smem, st>>>(tq, tkv, a);
  return cudaGetLastError();
}

}  // namespace mla
