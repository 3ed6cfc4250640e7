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
// Warp roles (320 threads, one CTA per SM):
//   warp 0      TMA producer: Q rows once per piece, then 9 boxes of 64 x 64
//               bf16 per 64-token page, 2-stage ring
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2..9  softmax, lazy rescale of O^T and the epilogue of each piece.
//               Query row r lives in TMEM lane 32*(r/16) + r%16. Each lane
//               quarter is read by two warps, one per 32-column half of the
//               score tile. The halves meet once per tile, in shared memory,
//               to agree on the row maximum.
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
constexpr int TC_THREADS = 320;              // warp 0 TMA, warp 1 MMA, warps 2..9 softmax
constexpr int TC_SM_THREADS = 256;
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
  float xmax[2][TC_ROWS];  // partial row maxima of the two column halves
  float xsum[TC_ROWS];     // row sum of the second column half
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

// 2^x with the hardware ex2 unit (max relative error about 2^-22); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
      mbar_init(&sm.s_empty[i], TC_SM_THREADS / 32);
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
      // Descriptor bases. Offsets inside the buffers are added to the
      // start-address field (bits 0-13, in 16-byte units); shared addresses
      // stay below 2^18 bytes, so the field never overflows.
      const uint64_t dQ = desc_kmajor(sm.q[0], 0);
      const uint64_t dP = desc_kmajor(sm.p, 0);
      uint64_t dK[TC_STAGES], dC[TC_STAGES];
      for (int s2 = 0; s2 < TC_STAGES; ++s2) {
        dK[s2] = desc_kmajor(sm.kv[s2][0], 0);
        dC[s2] = desc_ct(sm.kv[s2][0], 0);
      }
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
        const int s2 = pit % TC_STAGES;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = dC[s2] + ((2 * j * CHUNK_BYTES + kk * 2048) >> 4);
            const uint64_t bd = dP + ((kk * 32) >> 4);
            mma_bf16_ss(tmem + TM_O + 64 * j, ad, bd, idPV, (first && kk == 0) ? 0u : 1u);
          }
        }
        mma_commit(&sm.kv_empty[s2]);
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
          const int s2 = kv_it % TC_STAGES;
          if (!mbar_wait(&sm.kv_full[s2], (kv_it / TC_STAGES) & 1, WAIT_LIMIT)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4 * TC_KCH; ++k) {
            const uint32_t off = ((k >> 2) * CHUNK_BYTES + (k & 3) * 32) >> 4;
            mma_bf16_ss(tmem + TM_S + 64 * sb, dQ + off, dK[s2] + off, idS, k > 0 ? 1u : 0u);
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
    // ------------------------------------------------------------ softmax warps 2..9
    // A failed (timed-out) wait only sets `bad`. Every thread still passes
    // every named barrier, and the group leaves the loop together at the
    // end-of-tile barrier, so no barrier can be left half-filled.
    const int qd = warp & 3;                   // TMEM lane quarter this warp may access
    const int hf = (warp - 2) >> 2;            // score column half: [32*hf, 32*hf + 32)
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    const int row = 16 * qd + lane;            // score row held by this lane (lane < 16)
    const bool lane_has_row = lane < 16;
    const int tid_sm = threadIdx.x - 64;       // 0..255
    uint32_t kv_it = 0;
    int piece_idx = 0;
    bool abort = false;
    for (long long it = it_begin; it < it_end && !abort;) {
      const Piece pc = locate_piece(it, it_end, T_all, a.prefix, a.tiles, a.B);
      const int L = a.seq_lens[pc.b];
      const int rg = pc.g * a.RG + row;
      const int rows_valid = min(a.RG, rows_total - pc.g * a.RG);
      const bool row_ok = lane_has_row && row < rows_valid;
      const int pos_q = L - a.n_q + (row_ok ? rg / a.n_h : 0);
      float m = -INFINITY, l = 0.f;  // m: running max (shared by both halves); l: this half

      for (int i = 0; i < pc.n_tiles && !abort; ++i) {
        bool bad = false;
        const int t = pc.t_first + i;
        const int sb = kv_it & 1;
        const int s2 = kv_it % TC_STAGES;
        bad |= !mbar_wait(&sm.s_full[sb], (kv_it >> 1) & 1, WAIT_LIMIT);
        tc_fence_after();
        float sc[32];
        {
          float v[16];
          tmem_ld16(tmem + lane_base + TM_S + 64 * sb + 32 * hf, v);
#pragma unroll
          for (int k = 0; k < 16; ++k) sc[k] = v[k];
          tmem_ld16(tmem + lane_base + TM_S + 64 * sb + 32 * hf + 16, v);
#pragma unroll
          for (int k = 0; k < 16; ++k) sc[16 + k] = v[k];
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.s_empty[sb]);

        const int j0 = t * TC_TOK + 32 * hf;  // token of sc[0]
        if (row_ok && j0 + 31 <= L - a.n_q) {
#pragma unroll
          for (int c = 0; c < 32; ++c) sc[c] *= a.scale_log2;
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            sc[c] = (row_ok && j0 + c <= pos_q) ? sc[c] * a.scale_log2 : -INFINITY;
        }
        float pm[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          pm[u] = fmaxf(fmaxf(sc[4 * u], sc[4 * u + 1]), fmaxf(sc[4 * u + 2], sc[4 * u + 3]));
        const float pmax = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                 fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
        const bool first = (i == 0);
        if (lane_has_row) sm.xmax[hf][row] = pmax;
        // One barrier: publishes both halves' maxima and tells everyone
        // whether any row must rescale (or any wait failed).
        const bool flag = bad || (!first && row_ok && pmax > m + RESCALE_THRESHOLD);
        const bool any = named_bar_or(1, TC_SM_THREADS, flag);
        const float m_new =
            lane_has_row ? fmaxf(m, fmaxf(sm.xmax[0][row], sm.xmax[1][row])) : -INFINITY;
        const bool need = !first && row_ok && (m_new > m + RESCALE_THRESHOLD);
        const float m_use = (first || need) ? m_new : m;
        const float alpha = (m == -INFINITY || first) ? 0.f : fast_exp2(m - m_use);
        // A row with nothing visible yet keeps m_use = -inf; subtracting 0
        // instead maps its -inf scores to 2^-inf = 0 rather than NaN.
        const float m_sub = (m_use == -INFINITY) ? 0.f : m_use;

        // P buffer free and O^T stable once the previous value MMA has finished.
        if (kv_it > 0) bad |= !mbar_wait(&sm.p_empty, (kv_it - 1) & 1, WAIT_LIMIT);
        tc_fence_after();
        if (any) {
          if (named_bar_or(1, TC_SM_THREADS, bad)) {
            abort = true;
          } else {
            if (hf == 0 && lane_has_row) sm.row_alpha[row] = need ? alpha : 1.f;
            named_bar_sync(1, TC_SM_THREADS);
            for (int j = 2 * hf; j < 2 * hf + 2; ++j) {
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
        }
        // P half-row -> shared memory (bf16, 128B-swizzled K-major)
        if (lane_has_row && !abort) {
          float psum = 0.f;
          uint8_t* prow = sm.p + row * 128;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float x0 = sc[ch * 8 + 2 * k], x1 = sc[ch * 8 + 2 * k + 1];
              const float p0 = fast_exp2(x0 - m_sub), p1 = fast_exp2(x1 - m_sub);
              const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
              psum += __low2float(pb) + __high2float(pb);
              w[k] = *reinterpret_cast<const uint32_t*>(&pb);
            }
            const int unit = 4 * hf + ch;
            *reinterpret_cast<uint4*>(prow + ((unit ^ (row & 7)) * 16)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (row_ok) {
            l = l * alpha + psum;
            m = m_use;
          }
        }
        // Rows past the end of the sequence may hold anything; zero their
        // latent columns so that 0 * garbage cannot reach the accumulator.
        const int jt = t * TC_TOK;
        if (!abort && jt + TC_TOK > L) {
          const int r0 = L - jt;  // first invalid row in this tile
          const int nrow = TC_TOK - r0;
          for (int i2 = tid_sm; i2 < nrow * 8 * 8; i2 += TC_SM_THREADS) {
            const int rr = r0 + i2 / 64, ch = (i2 / 8) % 8, u = i2 % 8;
            *reinterpret_cast<uint4*>(sm.kv[s2][ch] + rr * 128 + u * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (named_bar_or(1, TC_SM_THREADS, bad)) abort = true;
        if (tid_sm == 0 && !abort) mbar_arrive(&sm.p_full);
        ++kv_it;
      }
      if (abort) break;

      // ---- epilogue of the piece: O^T / l -> workspace slot
      bool bad = !mbar_wait(&sm.o_full, piece_idx & 1, WAIT_LIMIT);
      tc_fence_after();
      if (hf == 1 && lane_has_row) sm.xsum[row] = l;
      if (named_bar_or(1, TC_SM_THREADS, bad)) {
        abort = true;
        break;
      }
      const int slot = blockIdx.x + pc.g * a.B + pc.b;
      if (hf == 0 && lane_has_row) {
        const float lt = l + sm.xsum[row];
        sm.row_inv_l[row] = (row_ok && lt > 0.f) ? 1.f / lt : 0.f;
        if (row_ok)
          a.part_lse[static_cast<size_t>(slot) * a.RG + row] =
              lt > 0.f ? (m + log2f(lt)) * 0.6931471805599453f : -INFINITY;
      }
      named_bar_sync(1, TC_SM_THREADS);
      float* dst = a.part_o + static_cast<size_t>(slot) * a.RG * 512;
      for (int j = 2 * hf; j < 2 * hf + 2; ++j) {
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
      named_bar_sync(1, TC_SM_THREADS);
      if (tid_sm == 0) mbar_arrive(&sm.o_empty);
      ++piece_idx;
      it += pc.n_tiles;
    }
    if (abort && tid_sm == 0) note_timeout(sm, a.err);
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

bool encode_rows_map(CUtensorMap* m, const void* base, uint64_t rows) {
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

// Tensor maps depend only on (base address, rows), so recent ones are kept.
struct MapCache {
  static constexpr int kSlots = 32;
  struct Entry {
    const void* base = nullptr;
    uint64_t rows = 0;
    CUtensorMap map;
  } e[kSlots];
  int next = 0;
  std::mutex mu;
};

bool make_rows_map(CUtensorMap* m, const void* base, uint64_t rows) {
  static MapCache cache;
  std::lock_guard<std::mutex> lk(cache.mu);
  for (auto& x : cache.e) {
    if (x.base == base && x.rows == rows) {
      *m = x.map;
      return true;
    }
  }
  if (!encode_rows_map(m, base, rows)) return false;
  auto& slot = cache.e[cache.next];
  cache.next = (cache.next + 1) % MapCache::kSlots;
  slot.base = base;
  slot.rows = rows;
  slot.map = *m;
  return true;
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
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  attend_tc_kernel<<<p.C, TC_THREADS, smem, st>>>(tq, tkv, a);
  return cudaGetLastError();
}

}  // namespace mla
