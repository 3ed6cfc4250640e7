// a3 (tensor-core variant): split-KV attention of absorbed queries over the
// paged latent cache, on tcgen05 / TMEM with TMA-staged tiles, one pair of
// CTAs (a 2-CTA cluster) per work range.
//
//   S   = Q K^T * scale        Q: [128 query rows x 576], K: [64 tokens x 576]
//   P   = online softmax of S (causal mask j <= pos_q)
//   O  += P C                  C: the 512 latent columns of the same tile
//
// Sources: "Multi-head Latent Attention: the KV cache, compressed", sections
// "Absorption: the part that makes it free" (queries are projected into
// latent space and dotted against the cache; keys are never built) and
// "RoPE, and why the explanations stop here" (the score is a content part
// plus a decoupled RoPE part, which one 576-wide dot product over
// [c | k_rope] computes); "Multi-head Latent Attention and KV Cache
// Compression", section "The absorption trick and decoupled RoPE" (the
// output is the softmax-weighted sum of latents, up-projected later).
//
// Why a CTA pair on sm_103a. All heads share one 576-wide key row and one
// 512-wide value row per token, so for 128 query rows both products are
// dense M = 128 contractions. The fp32 accumulator of 128 rows x 512 latent
// columns is 256 KB, the whole TMEM of one SM, with no room left for
// scores. So the two CTAs of a cluster split the columns: CTA r holds latent
// columns [256r, 256r + 256) and rotary columns [512 + 32r, 512 + 32r + 32)
// of every tile and of Q, and accumulates O for its 256 latent columns
// (256 TMEM columns). Each CTA computes a partial score over its 288
// columns (M = 128, N = 64, K = 288). The pair swaps the partials through
// distributed shared memory: one bulk copy per tile and direction that counts
// its bytes on the receiver's mbarrier. Each then adds the two partials. fp32
// addition is commutative, so both CTAs hold bit-identical scores, run the
// same softmax and agree on every row maximum and sum without further
// messages. Every cache byte is read from HBM once, by one CTA.
//
// The exchange is a pipeline stage of its own, so that its latency overlaps
// the softmax of the previous tile instead of adding to it:
//
//   TMA -> score MMA -> sender warps -> (peer) -> softmax warps -> value MMA
//
// TMEM (512 columns): two 64-column score slots (tile parity), a 32-column
// buffer for P (bf16 pairs, read by the value MMA straight from TMEM as its
// A operand), 96 columns of Q (192 of this CTA's latent columns) and the
// 256-column latent accumulator. The sender warps and the softmax warps
// both read a score slot; each rounds the CTA's partial to fp16 the same
// way, the senders for the peer and the softmax for its own half of the sum.
//
// The partials travel by the bulk-copy engine (cp.async.bulk from a local
// staging buffer into the peer's exchange buffer), not by st.async from
// registers: while a warp streams 16 KB of st.async, the other warps' TMEM
// loads and 16-byte shared loads on the SM wait behind it for about the
// length of the transfer, which stalled the softmax warps once per tile.
//
// Warp roles (512 threads, one CTA per SM):
//   warp 0      TMA producer: Q (1 + 1 boxes) once per piece, then per
//               64-token page the latent columns and the rotary box, 4-stage
//               ring
//   warp 1      TMEM allocator and value-MMA issuer
//   warps 2, 3  score-MMA issuers, warp 2 for even tiles, warp 3 for odd
//               tiles, each into its own score slot
//   warps 4..7  senders: warp w reads the score slot's lane quarter w % 4
//               (one query row per lane, all 64 tokens), rounds the partial
//               to fp16 and writes the fp16 words into the staging buffer,
//               from which one thread copies them to the peer. They also put
//               the TMEM part of Q in place at each piece.
//   warps 8..15 softmax: warp w reads lane quarter w % 4 and tokens
//               [32h, 32h + 32), h = (w - 8) / 4, rounds its own partial to
//               fp16 and adds the peer's with one mixed-precision add per
//               score.
//               The two warps of a lane quarter meet at a 64-thread named
//               barrier to agree on the row maximum. One set of warps handles
//               every tile, so the running max and row sums live in
//               registers.
//
// Work ranges. Each pair walks a contiguous range of (group, sequence, page)
// items from the plan; ranges are balanced by pages plus a charge per
// sequence piece (a piece change costs an epilogue and a Q load). The kernel
// is launched with programmatic dependent launch: its setup overlaps the end
// of the query-absorption kernel, and it reads nothing that kernel writes
// before griddepcontrol.wait.
//
// Lazy rescale: a row's running max is only raised when the new max exceeds
// it by more than 8 (log2 units). Otherwise P is computed against the stale
// max, so its entries stay <= 2^8. The final division by the row sum cancels
// the offset exactly.
//
// Every mbarrier wait is bounded. On a timeout the CTA sets
// MLA_DEVERR_TIMEOUT and stops issuing work. It still drains what it issued,
// meets its peer at the final cluster barrier, frees TMEM and returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cmath>
#include <mutex>

#include "device_common.cuh"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace mla {
namespace {

using namespace mla_ptx;

constexpr int TP_ROWS = 128;                  // query rows per group (MMA M)
constexpr int TP_TOK = 64;                    // tokens per tile = page size
constexpr int TP_STAGES = 4;
constexpr int TP_THREADS = 512;
constexpr int F8_CONV_WARP0 = 16;             // fp8 cache: first converter warp
constexpr int F8_CONV_WARPS = 4;
template <bool FP8>
constexpr int kThreads = FP8 ? TP_THREADS + 32 * F8_CONV_WARPS : TP_THREADS;
constexpr int TP_SEND_WARP0 = 4;              // first sender warp
constexpr int TP_SM_WARP0 = 8;                // first softmax warp
constexpr int TP_SM_WARPS = 8;
constexpr uint32_t QC_BOX = 128 * 128;        // 128 rows x 64 bf16, 128B swizzle
constexpr uint32_t QR_BOX = 128 * 64;         // 128 rows x 32 bf16, 64B swizzle
constexpr uint32_t KC_BOX = 64 * 128;         // 64 tokens x 64 bf16
constexpr uint32_t KR_BOX = 64 * 64;          // 64 tokens x 32 bf16
constexpr uint32_t Q_BYTES = QC_BOX + QR_BOX;   // Q through TMA (the rest goes to TMEM)
constexpr uint32_t STAGE_BYTES = 4 * KC_BOX + KR_BOX;
constexpr uint32_t X_BYTES = TP_ROWS * TP_TOK * 2;  // fp16 partial scores
constexpr uint32_t TM_S = 0;                  // score slots at columns 0 and 64
constexpr uint32_t TM_P = 128;                // P buffer, 32 columns
constexpr uint32_t TM_Q = 160;                // Q latent columns 64..255 of this CTA (bf16 pairs)
constexpr uint32_t TM_O = 256;                // latent accumulator, 256 columns
constexpr uint32_t SEND_BAR = 5;              // named barrier of the four sender warps
constexpr long long WAIT_LIMIT = 4000000000LL;  // ~2 s at 2 GHz
constexpr float RESCALE_THRESHOLD = 8.f;        // log2 units

// fp8 (e4m3) cache: per page and CTA, the latent codes of this CTA's 256
// columns, its 32 rotary codes and the page's 64 row scales arrive by TMA in
// a ring of F8_STAGES; the softmax warps convert them to fp16 (exact for
// every e4m3 value) into F8_KV_STAGES compute stages laid out like the bf16
// ones, two tiles ahead of the score MMAs.
constexpr int F8_STAGES = 2;
constexpr int F8_KV_STAGES = 3;
constexpr uint32_t F8C_BYTES = TP_TOK * 256;
constexpr uint32_t F8R_BYTES = TP_TOK * 32;
constexpr uint32_t F8_TX_BYTES = F8C_BYTES + F8R_BYTES + TP_TOK * 4;

struct __align__(128) F8Stage {
  uint8_t c[F8C_BYTES];  // [token][256 codes], no swizzle
  uint8_t r[F8R_BYTES];  // [token][32 codes]
  float s[TP_TOK];       // row scales of the page
};

template <bool FP8>
struct F8Part {
  F8Stage st[F8_STAGES];
  float kscale[F8_KV_STAGES][TP_TOK];   // row scales of a compute stage (0 past the end)
  float klscale[F8_KV_STAGES][TP_TOK];  // their log2 (-inf past the end)
  uint64_t full[F8_STAGES], empty[F8_STAGES];
};
template <>
struct F8Part<false> {};

template <bool FP8>
struct __align__(1024) PairSmemT {
  static constexpr int NS = FP8 ? F8_KV_STAGES : TP_STAGES;  // compute stages
  uint8_t qc[QC_BOX];  // Q latent columns 0..63 of this CTA's half
  uint8_t qr[QR_BOX];
  struct Stage {
    uint8_t c[4][KC_BOX];
    uint8_t r[KR_BOX];
  } kv[NS];
  // peer's partial scores, fp16 pairs: [buffer][row][64 tokens], 16-byte units swizzled
  uint32_t xbuf[2][TP_ROWS * TP_TOK / 2];
  // this CTA's partial scores of the tile being sent, same layout
  uint32_t sendbuf[TP_ROWS * TP_TOK / 2];
  F8Part<FP8> f8;
  uint64_t kv_full[NS], kv_empty[NS];
  uint64_t q_full, q_empty;
  uint64_t s_full[2], s_empty[2];   // score slot by tile parity
  uint64_t own_ready[2];            // the sender warps are done reading the slot
  uint64_t x_full[2], x_sendok[2];  // peer's partial arrived / peer's buffer free
  uint64_t p_full[2], pv_done[2];
  uint64_t o_full, o_empty;
  uint64_t drain[3];
  uint32_t tmem_base;
  int abort_flag;
  float xmax[2][2][TP_ROWS];   // [tile parity][column half] partial row maxima
  float st_l[2][TP_ROWS];      // [column half]: row sums at the end of a piece
};

static_assert(sizeof(PairSmemT<false>) + 1024 <= 227 * 1024, "bf16 pair smem above 227 KB");
static_assert(sizeof(PairSmemT<true>) + 1024 <= 227 * 1024, "fp8 pair smem above 227 KB");

struct PairArgs {
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* tiles;
  const int32_t* prefix;
  const long long* bounds;  // [P + 1] first work item of each pair's range
  const int32_t* first_b;   // [P] sequence of each range's first work item
  float* part_o;
  float* part_lse;
  const uint16_t* qabs;       // [q_rows][576] absorbed queries, bf16 or fp16 bits (the TMEM part of Q)
  const float* row_scale;     // fp8 cache: [num_blocks * 64] row scales
  uint32_t* err;
  long long q_rows;
  int num_blocks, max_blocks, B, n_q, n_h, G, P;
  int chunked;  // 1: a stage's latent boxes come as one 3-D box; 0: as four 2-D boxes
};

// One piece: consecutive tiles of one (group, sequence) inside a pair's range.
struct Piece {
  int g, b, t_first, n_tiles;
};

// The piece that starts at work item `it` of a range ending at `end`, found
// by stepping forward from sequence b0 of group g0, which lies at or before
// it (the plan's first sequence of the range, or the sequence after the
// previous piece). Without empty sequences in between that is one round of
// independent loads, not a search.
__device__ __noinline__ Piece piece_at(long long it, long long end, long long T_all,
                                      const PairArgs& a, int g0, int b0) {
  Piece pc;
  pc.g = static_cast<int>(it / T_all);
  const long long rem = it % T_all;
  int b = pc.g == g0 ? min(b0, a.B - 1) : 0;
  while (b + 1 < a.B && a.prefix[b + 1] <= rem) ++b;
  pc.b = b;
  pc.t_first = static_cast<int>(rem - a.prefix[b]);
  const long long stop =
      min(end, static_cast<long long>(pc.g) * T_all + a.prefix[b] + a.tiles[b]);
  pc.n_tiles = static_cast<int>(stop - it);
  return pc;
}

// Walks the tiles of a pair's range in order: kv counts tiles from 0, i is
// the index inside the current piece, piece counts pieces from 0. The
// range's invariants stay in the kernel parameters, not in registers.
struct TileCursor {
  long long it;
  int left;  // tiles left in the range, this one included
  Piece pc;
  int i, piece;
  uint32_t kv;
  __device__ void init(long long b, long long e, const PairArgs& a, int pair) {
    it = b;
    left = static_cast<int>(e - b);
    i = 0;
    piece = 0;
    kv = 0;
    if (left > 0) {
      const long long T_all = a.prefix[a.B];
      pc = piece_at(it, e, T_all, a, static_cast<int>(it / T_all), a.first_b[pair]);
    }
  }
  __device__ bool valid() const { return left > 0; }
  __device__ bool first() const { return i == 0; }
  __device__ bool last() const { return i == pc.n_tiles - 1; }
  __device__ int tile() const { return pc.t_first + i; }
  __device__ void next(const PairArgs& a) {
    ++it;
    --left;
    ++i;
    ++kv;
    if (i == pc.n_tiles) {
      i = 0;
      ++piece;
      if (left > 0) pc = piece_at(it, it + left, a.prefix[a.B], a, pc.g, pc.b + 1);
    }
  }
};

// 2^x with the hardware ex2 unit (max relative error about 2^-22); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <class SM>
__device__ __forceinline__ void note_timeout(SM& sm, uint32_t* err) {
  *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
  set_error(err, MLA_DEVERR_TIMEOUT);
}

template <class SM>
__device__ __forceinline__ bool aborted(SM& sm) {
  return *reinterpret_cast<volatile int*>(&sm.abort_flag) != 0;
}

// Partial score (already in log2 units) -> fp16, round to nearest. Scores
// beyond the fp16 range saturate to +-65504 instead of becoming inf.
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float2 unpack_half2(uint32_t u) {
  return __half22float2(*reinterpret_cast<const __half2*>(&u));
}

// (fp32) of the low / high fp16 half of u, plus c0 / c1, rounded once: the
// fp16 value converts exactly, so this is the fp32 sum of the two values.
__device__ __forceinline__ float2 add_half2_f32(uint32_t u, float c0, float c1) {
  float d0, d1;
  asm("{\n\t.reg .f16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.f16 %0, lo, %3;\n\t"
      "add.rn.f32.f16 %1, hi, %4;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "r"(u), "f"(c0), "f"(c1));
  return make_float2(d0, d1);
}

// Byte offset of 16-byte unit u (0..7) of query row `row` in an exchange buffer.
__device__ __forceinline__ uint32_t xoff(int row, int u) {
  return static_cast<uint32_t>(row * 128 + ((u ^ (row & 7)) * 16));
}

// Sender side of tile kv, for query row `row` (one per lane of the warp's
// lane quarter): reads this CTA's partial scores of all 64 tokens from the
// score slot (the queries carry scale * log2(e), so they are in log2
// units), rounds them to fp16 and writes the fp16 words into the staging
// buffer. (This CTA's softmax reads the slot itself and rounds the same
// way.) The leader thread then copies the staged tile into the peer's
// exchange buffer kv & 1 with one bulk copy that counts its bytes on the
// peer's mbarrier. `bad` carries this thread's earlier timeouts. Returns
// SEND_STOP in all 128 sender threads if any of them had timed out (then
// this tile is not processed), SEND_LATE in the leader if its wait for the
// peer's buffer timed out here (then nothing was sent), else SEND_OK.
enum SendResult { SEND_OK = 0, SEND_LATE = 1, SEND_STOP = 2 };
template <class SM>
__device__ __forceinline__ SendResult send_tile(SM& sm, uint32_t slot, int row, int lane,
                                                bool leader, uint32_t kv, uint32_t peer,
                                                bool bad) {
  const int b = kv & 1;
  bad |= !mbar_wait(&sm.s_full[b], (kv >> 1) & 1, WAIT_LIMIT);
  // The previous tile's copy has to be done reading the staging buffer.
  if (leader && kv > 0) bulk_wait_read_all();
  if (named_bar_or(SEND_BAR, 128, bad)) return SEND_STOP;
  tc_fence_after();
  uint32_t h0[16], h1[16];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float v0[16], v1[16];
    tmem_ld16(slot + 32 * half, v0);
    tmem_ld16(slot + 32 * half + 16, v1);
    tmem_wait_ld();
    uint32_t (&h)[16] = half ? h1 : h0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      h[k] = pack_half2(v0[2 * k], v0[2 * k + 1]);
      h[8 + k] = pack_half2(v1[2 * k], v1[2 * k + 1]);
    }
  }
  const uint32_t stg = smem_u32(sm.sendbuf);
#pragma unroll
  for (int u = 0; u < 4; ++u)
    st_shared_v4(stg + xoff(row, u), h0[4 * u], h0[4 * u + 1], h0[4 * u + 2], h0[4 * u + 3]);
#pragma unroll
  for (int u = 0; u < 4; ++u)
    st_shared_v4(stg + xoff(row, 4 + u), h1[4 * u], h1[4 * u + 1], h1[4 * u + 2], h1[4 * u + 3]);
  fence_proxy_async_smem();  // the staged words are read by the bulk copy
  tc_fence_before();
  named_bar_sync(SEND_BAR, 128);
  if (lane == 0) mbar_arrive(&sm.own_ready[b]);
  bool late = false;
  if (leader) {
    // The peer's buffer kv & 1 is free once it has consumed tile kv - 2.
    if (kv >= 2) late = !mbar_wait(&sm.x_sendok[b], ((kv >> 1) - 1) & 1, WAIT_LIMIT);
    // this CTA's buffer kv & 1 expects the peer's copy of the same tile
    mbar_arrive_expect_tx(&sm.x_full[b], X_BYTES);
    if (!late) {
      bulk_copy_to_peer(mapa_shared(smem_u32(sm.xbuf[b]), peer), sm.sendbuf, X_BYTES,
                        mapa_shared(smem_u32(&sm.x_full[b]), peer));
      bulk_commit();
    }
  }
  return late ? SEND_LATE : SEND_OK;
}

// The sender warps put this CTA's Q latent columns 64..255 of the piece's
// 128 query rows into TMEM (bf16 pairs, row per lane), where the score MMAs
// read them as their A operand, once the previous piece's score MMAs are
// done with them. Rows past the end of the queries are zero. Returns true on
// timeout.
template <class SM>
__device__ __forceinline__ bool load_q_tmem(SM& sm, const PairArgs& a, uint32_t tmem,
                                            uint32_t lane_base, int row, int lane, uint32_t rank,
                                            const TileCursor& cur) {
  bool bad = false;
  if (cur.piece > 0) bad = !mbar_wait(&sm.q_empty, (cur.piece - 1) & 1, WAIT_LIMIT);
  tc_fence_after();
  const long long grow =
      static_cast<long long>(cur.pc.b) * a.n_q * a.n_h + cur.pc.g * TP_ROWS + row;
  const uint4* src = reinterpret_cast<const uint4*>(a.qabs + grow * 576 + 256 * rank + 64);
  const bool in = grow < a.q_rows;
#pragma unroll
  for (int j = 0; j < 6; ++j) {
    uint32_t w[16];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint4 v = in ? src[4 * j + u] : make_uint4(0, 0, 0, 0);
      w[4 * u] = v.x;
      w[4 * u + 1] = v.y;
      w[4 * u + 2] = v.z;
      w[4 * u + 3] = v.w;
    }
    tmem_st16u(tmem + lane_base + TM_Q + 16 * j, w);
  }
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&sm.q_full);
  return bad;
}

// 16 e4m3 codes (one 16-byte unit, lowest address first) -> 16 fp16 values
// in eight f16x2 words, same order. Every e4m3 value is exact in fp16.
__device__ __forceinline__ void e4m3x16_to_f16(const uint4& v, uint32_t (&w)[8]) {
  const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
        static_cast<__nv_fp8x2_storage_t>(in[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
        static_cast<__nv_fp8x2_storage_t>(in[i] >> 16), __NV_E4M3);
    w[2 * i] = static_cast<uint32_t>(lo.x) | (static_cast<uint32_t>(lo.y) << 16);
    w[2 * i + 1] = static_cast<uint32_t>(hi.x) | (static_cast<uint32_t>(hi.y) << 16);
  }
}

// fp8 cache: the converter warps (thread ctid of NTHR) convert tile cv.kv
// from its e4m3 ring stage into its fp16 compute stage, in the layout the TMA
// gives the bf16 stages (four 128-byte-swizzled latent boxes, one
// 64-byte-swizzled rotary box), and copy the page's row scales (and their
// log2) beside it. Rows past the sequence's end become zeros with scale 0,
// whatever the cache holds there. Each warp then arrives on the compute
// stage's full barrier and the ring stage's empty barrier. Returns false on
// a timeout (nothing converted, nothing arrived).
template <int NTHR, class SM>
__device__ __forceinline__ bool convert_tile(SM& sm, const PairArgs& a, const TileCursor& cv,
                                             int ctid, int lane) {
  const uint32_t j = cv.kv;
  const int s8 = j % F8_STAGES, sc = j % F8_KV_STAGES;
  bool ok = true;
  // the compute stage is free once the value MMAs of tile j - 3 are done
  if (j >= F8_KV_STAGES)
    ok = mbar_wait(&sm.kv_empty[sc], ((j / F8_KV_STAGES) - 1) & 1, WAIT_LIMIT);
  ok = ok && mbar_wait(&sm.f8.full[s8], (j / F8_STAGES) & 1, WAIT_LIMIT);
  if (!__all_sync(0xffffffffu, ok)) return false;
  const int L = a.seq_lens[cv.pc.b];
  const int valid = min(TP_TOK, max(0, L - cv.tile() * TP_TOK));
  const F8Stage& f = sm.f8.st[s8];
  auto& dst = sm.kv[sc];
  constexpr int kUnits = 18;  // 16-byte input units per row: 16 latent, 2 rotary
  static_assert(NTHR % 32 == 0, "warps take whole 32-item groups");
  for (int k = ctid; k < TP_TOK * kUnits; k += NTHR) {
    // Latent items go in 8-thread phases over rows 2 rp and 2 rp + 1: the
    // first row's four units of box bsel, the second's of box bsel ^ 1. Their
    // loads and both stores then fall in eight different 16-byte bank
    // groups (the rows' swizzles differ in the low bit). Rotary items follow.
    int r, u;
    if (k < TP_TOK * 16) {
      const int rp = k >> 5, bsel = (k >> 3) & 3, t = k & 7, rr = t >> 2;
      r = 2 * rp + rr;
      u = 4 * (bsel ^ rr) + (t & 3);
    } else {
      const int kk = k - TP_TOK * 16;
      r = kk >> 1;
      u = 16 + (kk & 1);
    }
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < valid)
      v = u < 16 ? *reinterpret_cast<const uint4*>(f.c + r * 256 + u * 16)
                 : *reinterpret_cast<const uint4*>(f.r + r * 32 + (u - 16) * 16);
    uint32_t w[8];
    e4m3x16_to_f16(v, w);
    uint8_t* row;
    int ua, ub;
    if (u < 16) {  // latent box u / 4, 16-byte units 2 (u % 4) and 2 (u % 4) + 1 of 8
      row = dst.c[u >> 2] + r * 128;
      const int u0 = 2 * (u & 3);
      ua = u0 ^ (r & 7);
      ub = (u0 + 1) ^ (r & 7);
    } else {  // rotary box, units 2 (u - 16) and 2 (u - 16) + 1 of 4
      row = dst.r + r * 64;
      const int u0 = 2 * (u - 16), x = (r >> 1) & 3;
      ua = u0 ^ x;
      ub = (u0 + 1) ^ x;
    }
    *reinterpret_cast<uint4*>(row + ua * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(row + ub * 16) = make_uint4(w[4], w[5], w[6], w[7]);
  }
  for (int k = ctid; k < TP_TOK; k += NTHR) {
    const bool in = k < valid;
    const float sv = in ? f.s[k] : 0.f;
    sm.f8.kscale[sc][k] = sv;
    sm.f8.klscale[sc][k] = in ? __log2f(sv) : -INFINITY;
  }
  fence_proxy_async_smem();  // the converted tile is read by the MMAs
  __syncwarp();
  if (lane == 0) {
    mbar_arrive(&sm.kv_full[sc]);
    mbar_arrive(&sm.f8.empty[s8]);
  }
  return true;
}

template <bool FP8>
__global__ void __launch_bounds__(kThreads<FP8>, 1)
attend_tc_kernel(const __grid_constant__ CUtensorMap tmap_qc,
                 const __grid_constant__ CUtensorMap tmap_qr,
                 const __grid_constant__ CUtensorMap tmap_kc,
                 const __grid_constant__ CUtensorMap tmap_kr, PairArgs a) {
  using Smem = PairSmemT<FP8>;
  constexpr int NS = Smem::NS;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int pair = static_cast<int>(cluster_id_x());

  // Setup first: with programmatic dependent launch it overlaps the end of
  // the query-absorption kernel, whose outputs are read only after the wait.
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      // bf16: the TMA's bytes; fp8: the converter warps
      mbar_init(&sm.kv_full[s], FP8 ? F8_CONV_WARPS : 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    if constexpr (FP8) {
      for (int s = 0; s < F8_STAGES; ++s) {
        mbar_init(&sm.f8.full[s], 1);
        mbar_init(&sm.f8.empty[s], F8_CONV_WARPS);
      }
    }
    mbar_init(&sm.q_full, 1 + 4);  // TMA bytes + the four sender warps' TMEM part
    mbar_init(&sm.q_empty, 2);     // one commit from each score-MMA issuer
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_empty[i], TP_SM_WARPS);
      mbar_init(&sm.own_ready[i], 4);
      mbar_init(&sm.x_full[i], 1);
      mbar_init(&sm.x_sendok[i], TP_SM_WARPS);
      mbar_init(&sm.p_full[i], TP_SM_WARPS);
      mbar_init(&sm.pv_done[i], 1);
    }
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.o_empty, TP_SM_WARPS);
    for (int i = 0; i < 3; ++i) mbar_init(&sm.drain[i], 1);
    sm.abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync();  // both CTAs' barriers exist before either arrives remotely
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  griddep_wait();
  griddep_launch_dependents();
  const long long T_all = a.prefix[a.B];
  const long long N = T_all * a.G;
  // Both CTAs of a pair see the same range, so they skip the work together.
  const long long it_begin = N > 0 ? a.bounds[pair] : 0;
  const long long it_end = N > 0 ? a.bounds[pair + 1] : 0;
  const int rows_total = a.n_q * a.n_h;

  if (it_begin >= it_end) {
    // empty range: straight to the final cluster barrier
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmap_qc);
      prefetch_tmap(&tmap_qr);
      prefetch_tmap(&tmap_kc);
      prefetch_tmap(&tmap_kr);
      // With one 128-row group per sequence every page is read once: stream
      // it past L2. With several (two query tokens, prefill chunks) each group
      // reads the page again, and the pairs walking the other groups read it
      // at about the same time: keep it in L2.
      const uint64_t pol = a.G > 1 ? policy_evict_normal() : policy_evict_first();
      const int xr = 512 + 32 * static_cast<int>(rank);
      uint32_t kv_it = 0;
      int piece_idx = 0;
      constexpr int RING = FP8 ? F8_STAGES : TP_STAGES;  // stages the TMA fills
      uint32_t issued[RING] = {};
      bool stop = false;
      int prev_g = static_cast<int>(it_begin / T_all), next_b = a.first_b[pair];
      for (long long it = it_begin; it < it_end && !stop && !aborted(sm);) {
        const Piece pc = piece_at(it, it_end, T_all, a, prev_g, next_b);
        prev_g = pc.g;
        next_b = pc.b + 1;
        if (piece_idx > 0 && !mbar_wait(&sm.q_empty, (piece_idx - 1) & 1, WAIT_LIMIT)) {
          note_timeout(sm, a.err);
          break;
        }
        const int qrow0 = pc.b * rows_total + pc.g * TP_ROWS;
        mbar_arrive_expect_tx(&sm.q_full, Q_BYTES);
        tma_load_2d(sm.qc, &tmap_qc, 256 * static_cast<int>(rank), qrow0, &sm.q_full);
        tma_load_2d(sm.qr, &tmap_qr, xr, qrow0, &sm.q_full);
        const int32_t* pt = a.page_table + static_cast<size_t>(pc.b) * a.max_blocks;
        int page_next = pt[pc.t_first];
        for (int t = pc.t_first; t < pc.t_first + pc.n_tiles; ++t) {
          int page = page_next;
          if (t + 1 < pc.t_first + pc.n_tiles) page_next = pt[t + 1];
          const int s = kv_it % RING;
          const uint32_t n = kv_it / RING;
          uint64_t* empty_bar;
          if constexpr (FP8) empty_bar = &sm.f8.empty[s];
          else empty_bar = &sm.kv_empty[s];
          if (kv_it >= RING && !mbar_wait(empty_bar, (n - 1) & 1, WAIT_LIMIT)) {
            note_timeout(sm, a.err);
            stop = true;
            break;
          }
          if (page < 0 || page >= a.num_blocks) {
            set_error(a.err, MLA_DEVERR_PAGE_RANGE);
            page = 0;
          }
          if constexpr (FP8) {
            // this CTA's 256 latent codes and 32 rotary codes of the page's
            // 64 rows, and the page's 64 row scales
            mbar_arrive_expect_tx(&sm.f8.full[s], F8_TX_BYTES);
            tma_load_2d_hint(sm.f8.st[s].c, &tmap_kc, 256 * static_cast<int>(rank),
                             page * TP_TOK, &sm.f8.full[s], pol);
            tma_load_2d_hint(sm.f8.st[s].r, &tmap_kr, xr, page * TP_TOK, &sm.f8.full[s], pol);
            bulk_load(sm.f8.st[s].s, a.row_scale + static_cast<size_t>(page) * TP_TOK,
                      TP_TOK * 4, &sm.f8.full[s]);
          } else {
            mbar_arrive_expect_tx(&sm.kv_full[s], STAGE_BYTES);
            if (a.chunked) {
              tma_load_3d_hint(sm.kv[s].c[0], &tmap_kc, 0, page * TP_TOK,
                               4 * static_cast<int>(rank), &sm.kv_full[s], pol);
            } else {
              for (int j = 0; j < 4; ++j)
                tma_load_2d_hint(sm.kv[s].c[j], &tmap_kc, 256 * static_cast<int>(rank) + 64 * j,
                                 page * TP_TOK, &sm.kv_full[s], pol);
            }
            tma_load_2d_hint(sm.kv[s].r, &tmap_kr, xr, page * TP_TOK, &sm.kv_full[s], pol);
          }
          ++issued[s];
          ++kv_it;
        }
        ++piece_idx;
        it += pc.n_tiles;
      }
      // Never leave a TMA write in flight past the end of the CTA.
      for (int s = 0; s < RING; ++s) {
        if (issued[s] == 0) continue;
        if constexpr (FP8) mbar_wait(&sm.f8.full[s], (issued[s] - 1) & 1, WAIT_LIMIT);
        else mbar_wait(&sm.kv_full[s], (issued[s] - 1) & 1, WAIT_LIMIT);
      }
      if (piece_idx > 0) mbar_wait(&sm.q_full, (piece_idx - 1) & 1, WAIT_LIMIT);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ value-MMA issuer
    // O (this CTA's 256 latent columns) += P C, with P read from TMEM.
    // pv_done[t & 1] tells the softmax when the P buffer and O are free.
    if (lane == 0) {
      const uint32_t idPV = FP8 ? idesc_f16_f32(128, 256, false, true)
                                : idesc_bf16_f32(128, 256, false, true);
      // C as the MN-major B operand: latent columns are contiguous (64 per
      // 128-byte row, the next 64 one box further), tokens step 128 B,
      // 8-token groups are 1024 B apart.
      const uint64_t dC0 = smem_desc(smem_u32(sm.kv[0].c[0]), KC_BOX, 1024, kSwizzle128B);
      constexpr uint32_t kStageDesc = sizeof(typename Smem::Stage) >> 4;  // stage stride, 16-B units
      bool ok = true;
      TileCursor cur;
      cur.init(it_begin, it_end, a, pair);
      for (; cur.valid() && ok; cur.next(a)) {
        const uint32_t t = cur.kv;
        if (!mbar_wait(&sm.p_full[t & 1], (t >> 1) & 1, WAIT_LIMIT)) { ok = false; break; }
        if (cur.first() && cur.piece > 0 &&
            !mbar_wait(&sm.o_empty, (cur.piece - 1) & 1, WAIT_LIMIT)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int s = t % NS;
        const uint32_t pcol = tmem + TM_P;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ts(tmem + TM_O, pcol + 8 * kk, dC0 + s * kStageDesc + ((2048u * kk) >> 4), idPV,
                      (cur.first() && kk == 0) ? 0u : 1u);
        mma_commit(&sm.kv_empty[s]);
        mma_commit(&sm.pv_done[t & 1]);
        if (cur.last()) mma_commit(&sm.o_full);
      }
      if (!ok) note_timeout(sm, a.err);
      // Every MMA issued above completes before TMEM is freed.
      mma_commit(&sm.drain[0]);
      mbar_wait(&sm.drain[0], 0, WAIT_LIMIT);
    }
  } else if (warp < TP_SEND_WARP0) {
    // ------------------------------------------------------------ score-MMA issuers
    // Warp 2 issues the even tiles into score slot 0, warp 3 the odd tiles
    // into slot 1, each as one accumulation of 18 K-steps: latent steps 0..3
    // with Q from shared memory, 4..15 with Q from TMEM, then the two rotary
    // steps. Two issuers keep the tensor pipe fed while either waits.
    if (lane == 0) {
      const uint32_t half = static_cast<uint32_t>(warp - 2);  // tile parity
      const uint32_t idS = FP8 ? idesc_f16_f32(128, TP_TOK, false, false)
                               : idesc_bf16_f32(128, TP_TOK, false, false);
      const uint64_t dQc = smem_desc(smem_u32(sm.qc), 16, 1024, kSwizzle128B);
      const uint64_t dQr = smem_desc(smem_u32(sm.qr), 16, 512, kSwizzle64B);
      const uint64_t dKc0 = smem_desc(smem_u32(sm.kv[0].c[0]), 16, 1024, kSwizzle128B);
      const uint64_t dKr0 = smem_desc(smem_u32(sm.kv[0].r), 16, 512, kSwizzle64B);
      constexpr uint32_t kStageDesc = sizeof(typename Smem::Stage) >> 4;  // stage stride, 16-B units
      const uint32_t dS = tmem + TM_S + 64 * half;
      bool ok = true;
      TileCursor cur;
      cur.init(it_begin, it_end, a, pair);
      while (cur.valid() && ok) {
        // one piece: wait for its Q, issue this parity's tiles, release Q
        if (!mbar_wait(&sm.q_full, cur.piece & 1, WAIT_LIMIT)) { ok = false; break; }
        tc_fence_after();
        const int piece = cur.piece;
        for (; cur.valid() && cur.piece == piece; cur.next(a)) {
          const uint32_t t = cur.kv;
          if ((t & 1) != half) continue;
          if (t >= 2 && !mbar_wait(&sm.s_empty[half], ((t >> 1) - 1) & 1, WAIT_LIMIT)) {
            ok = false;
            break;
          }
          const int s = t % NS;
          if (!mbar_wait(&sm.kv_full[s], (t / NS) & 1, WAIT_LIMIT)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dK = dKc0 + s * kStageDesc;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16_ss(dS, dQc + ((32u * k) >> 4), dK + ((32u * k) >> 4), idS, k > 0 ? 1u : 0u);
#pragma unroll
          for (int k = 4; k < 16; ++k) {
            const uint32_t koff = (KC_BOX * (k >> 2) + 32 * (k & 3)) >> 4;
            mma_bf16_ts(dS, tmem + TM_Q + 8 * (k - 4), dK + koff, idS, 1u);
          }
#pragma unroll
          for (int k = 0; k < 2; ++k)
            mma_bf16_ss(dS, dQr + ((32u * k) >> 4), dKr0 + s * kStageDesc + ((32u * k) >> 4), idS,
                        1u);
          mma_commit(&sm.s_full[half]);
        }
        if (!ok) break;
        mma_commit(&sm.q_empty);
      }
      if (!ok) note_timeout(sm, a.err);
      mma_commit(&sm.drain[1 + half]);
      mbar_wait(&sm.drain[1 + half], 0, WAIT_LIMIT);
    }
  } else if (warp < TP_SM_WARP0) {
    // ------------------------------------------------------------ sender warps 4..7
    const int qd = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    const int row = 32 * qd + lane;
    const bool leader = warp == TP_SEND_WARP0 && lane == 0;
    bool bad = false;
    TileCursor cur;
    cur.init(it_begin, it_end, a, pair);
    // The four warps meet at named barriers inside send_tile, which merge
    // their timeout flags, so they leave the loop together.
    for (; cur.valid(); cur.next(a)) {
      if (cur.first()) bad |= load_q_tmem(sm, a, tmem, lane_base, row, lane, rank, cur);
      const uint32_t kv = cur.kv;
      const SendResult r = send_tile(sm, tmem + lane_base + TM_S + 64 * (kv & 1), row, lane,
                                     leader, kv, peer, bad);
      bad = r != SEND_OK;
      if (r == SEND_STOP) break;
    }
    if (leader) bulk_wait_all();  // the last copies land before the peer may leave
    if (bad && lane == 0) note_timeout(sm, a.err);
  } else if (warp >= F8_CONV_WARP0) {
    // ------------------------------------------------------------ fp8 converter warps 16..19
    // Each tile as soon as its codes have landed and its compute stage is
    // free, independently of the other roles (no named barriers here).
    if constexpr (FP8) {
      const int ctid = (warp - F8_CONV_WARP0) * 32 + lane;
      TileCursor cv;
      cv.init(it_begin, it_end, a, pair);
      bool bad = false;
      for (; cv.valid() && !bad && !aborted(sm); cv.next(a))
        bad = !convert_tile<32 * F8_CONV_WARPS>(sm, a, cv, ctid, lane);
      if (bad && lane == 0) note_timeout(sm, a.err);
    }
  } else {
    // ------------------------------------------------------------ softmax warps 8..15
    // Warp w reads TMEM lane quarter w % 4 (query rows 32 (w % 4) .. +31, one
    // row per lane) and tokens [32 hh, 32 hh + 32), hh = (w - 8) / 4. The two
    // warps of a lane quarter agree on the row maximum at a 64-thread named
    // barrier; each keeps the sum of its half rows, referred to the running
    // max m, which both hold in registers.
    const int sw = warp - TP_SM_WARP0;          // 0..7
    const int hh = sw >> 2;
    const int qd = warp & 3;
    const uint32_t bar_id = 1 + qd;             // 64-thread barrier of the two halves
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    const int row = 32 * qd + lane;
    const int gtid = sw * 32 + lane;            // 0..255
    TileCursor cur;
    cur.init(it_begin, it_end, a, pair);
    float l = 0.f, m = -INFINITY;
    int L = 0, rows_valid = 0, pos_q = 0;
    bool row_ok = false, bad = false;
    // The two warps of a lane quarter leave the loop together, right after a
    // pair barrier has merged their timeout flags, so neither can be left
    // waiting at a named barrier.
    for (; cur.valid(); cur.next(a)) {
      const uint32_t kv = cur.kv;
      const int b = kv & 1;
      const bool first = cur.first();
      if (first) {
        l = 0.f;
        m = -INFINITY;
        L = a.seq_lens[cur.pc.b];
        rows_valid = min(TP_ROWS, rows_total - cur.pc.g * TP_ROWS);
        row_ok = row < rows_valid;
        pos_q = L - a.n_q + (row_ok ? (cur.pc.g * TP_ROWS + row) / a.n_h : 0);
      }
      const int t = cur.tile();
      const int s2 = kv % NS;

      // 1. full scaled scores = own partial (score slot) rounded to fp16 +
      // the peer's fp16 partial (exchange buffer): both CTAs add the same two
      // fp16 values, so they hold bit-identical scores
      bad |= !mbar_wait(&sm.own_ready[b], (kv >> 1) & 1, WAIT_LIMIT);
      bad |= !mbar_wait(&sm.x_full[b], (kv >> 1) & 1, WAIT_LIMIT);
      bad = __any_sync(0xffffffffu, bad);
      tc_fence_after();
      float sc[32];
      {
        float ow[2][16];
        tmem_ld16(tmem + lane_base + TM_S + 64 * b + 32 * hh, ow[0]);
        tmem_ld16(tmem + lane_base + TM_S + 64 * b + 32 * hh + 16, ow[1]);
        const uint8_t* xin = reinterpret_cast<const uint8_t*>(sm.xbuf[b]);
        uint4 pv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          pv[u] = *reinterpret_cast<const uint4*>(xin + xoff(row, 4 * hh + u));
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t pw[4] = {pv[u].x, pv[u].y, pv[u].z, pv[u].w};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int c = 8 * u + 2 * w;
            const float2 o = unpack_half2(pack_half2(ow[c >> 4][c & 15], ow[c >> 4][(c & 15) + 1]));
            const float2 x = add_half2_f32(pw[w], o.x, o.y);
            sc[c] = x.x;
            sc[c + 1] = x.y;
          }
        }
      }
      if constexpr (FP8) {
        // x_j = q . code_j; the score is scale_j x_j. (The scales were
        // written by these warps, released on the stage's full barrier.)
        bad |= !mbar_wait(&sm.kv_full[s2], (kv / NS) & 1, WAIT_LIMIT);
        const float* ks = sm.f8.kscale[s2] + 32 * hh;
#pragma unroll
        for (int c = 0; c < 32; ++c) sc[c] *= ks[c];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.s_empty[b]);  // the score slot may take tile kv + 2
        // At the end of a piece the epilogue borrows this exchange buffer, so
        // the peer may only refill it afterwards.
        if (!cur.last()) mbar_arrive_remote_relaxed(mapa_shared(smem_u32(&sm.x_sendok[b]), peer));
      }

      // 2. causal mask, row max (both halves), running max
      const int j0 = t * TP_TOK + 32 * hh;  // token of sc[0]
      if (!(row_ok && j0 + 31 <= L - a.n_q)) {
#pragma unroll
        for (int c = 0; c < 32; ++c) sc[c] = (row_ok && j0 + c <= pos_q) ? sc[c] : -INFINITY;
      }
      if constexpr (FP8) {
        // The running max tracks s_j + log2(scale_j), so that the value
        // weights p_j scale_j stay below 2^8 (fp16 range); l keeps the sum
        // of p_j itself. Any common reference cancels in O / l.
        const float* kl = sm.f8.klscale[s2] + 32 * hh;
        float pm = -INFINITY;
#pragma unroll
        for (int c = 0; c < 32; ++c) pm = fmaxf(pm, sc[c] + kl[c]);
        sm.xmax[b][hh][row] = pm;
      } else {
        float pm[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          pm[u] = fmaxf(fmaxf(fmaxf(sc[8 * u], sc[8 * u + 1]), fmaxf(sc[8 * u + 2], sc[8 * u + 3])),
                        fmaxf(fmaxf(sc[8 * u + 4], sc[8 * u + 5]), fmaxf(sc[8 * u + 6], sc[8 * u + 7])));
        sm.xmax[b][hh][row] = fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
      }
      if (named_bar_or(bar_id, 64, bad)) {
        bad = true;
        break;
      }
      const float pmax = fmaxf(sm.xmax[b][0][row], sm.xmax[b][1][row]);
      const float m_old = m;
      const float m_new = fmaxf(m_old, pmax);
      const bool need = !first && row_ok && (m_new > m_old + RESCALE_THRESHOLD);
      const float m_use = (first || need) ? m_new : m_old;
      // A row with nothing visible yet keeps m_use = -inf; subtracting 0
      // instead maps its -inf scores to 2^-inf = 0 rather than NaN.
      const float m_sub = (m_use == -INFINITY) ? 0.f : m_use;

      // 3. P (bf16 pairs; fp8 cache: p_j scale_j in fp16 pairs) into the
      // TMEM buffer, once the previous tile's value MMA has read it
      {
        float psum = 0.f;
        uint32_t w[16];
        const float* ks = nullptr;
        if constexpr (FP8) ks = sm.f8.kscale[s2] + 32 * hh;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float p0 = fast_exp2(sc[2 * k] - m_sub);
          const float p1 = fast_exp2(sc[2 * k + 1] - m_sub);
          psum += p0 + p1;
          if constexpr (FP8) {
            const __half2 ph = __floats2half2_rn(p0 * ks[2 * k], p1 * ks[2 * k + 1]);
            w[k] = *reinterpret_cast<const uint32_t*>(&ph);
          } else {
            const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
            w[k] = *reinterpret_cast<const uint32_t*>(&pb);
          }
        }
        if (kv >= 1)
          bad |= !mbar_wait(&sm.pv_done[(kv - 1) & 1], ((kv - 1) >> 1) & 1, WAIT_LIMIT);
        bad = __any_sync(0xffffffffu, bad);
        tc_fence_after();
        if (!bad) tmem_st16u(tmem + lane_base + TM_P + 16 * hh, w);
        tmem_wait_st();
        if (row_ok) l = (m_old == -INFINITY) ? psum : l * fast_exp2(m_old - m_use) + psum;
        m = m_use;
      }
      // 4. lazy rescale of this warp's rows of O (its half of the columns);
      // the previous tile's value MMA is done with O (waited for above)
      if (__any_sync(0xffffffffu, need)) {
        if (!bad) {
          const float f = need ? fast_exp2(m_old - m_use) : 1.f;
          for (int c0 = 0; c0 < 128; c0 += 16) {
            float v[16];
            const uint32_t ta = tmem + lane_base + TM_O + 128 * hh + c0;
            tmem_ld16(ta, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] *= f;
            tmem_st16(ta, v);
          }
          tmem_wait_st();
        }
      }

      // Rows past the end of the sequence may hold anything; zero their
      // latent columns so that 0 * garbage cannot reach the accumulator.
      // (The fp8 conversion already wrote zeros there.)
      const int jt = t * TP_TOK;
      if (!FP8 && jt + TP_TOK > L) {
        const int r0 = max(L - jt, 0);            // first invalid row in this tile
        const int n16 = (TP_TOK - r0) * 4 * 8;    // rows x boxes x 16-byte units
        for (int i2 = gtid; i2 < n16; i2 += TP_SM_WARPS * 32) {
          const int rr = r0 + i2 / 32, box = (i2 / 8) % 4, u = i2 % 8;
          *reinterpret_cast<uint4*>(sm.kv[s2].c[box] + rr * 128 + u * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[b]);

      if (cur.last()) {
        // ---- epilogue of the piece: O / l -> workspace slot
        sm.st_l[hh][row] = l;
        if (named_bar_or(bar_id, 64, bad)) bad = true;
        bad |= !mbar_wait(&sm.o_full, cur.piece & 1, WAIT_LIMIT);
        bad = __any_sync(0xffffffffu, bad);
        tc_fence_after();
        const float lt = sm.st_l[0][row] + sm.st_l[1][row];
        const float inv_l = (row_ok && lt > 0.f) ? 1.f / lt : 0.f;
        const int slot = pair + cur.pc.g * a.B + cur.pc.b;
        if (rank == 0 && hh == 0 && row_ok)
          a.part_lse[static_cast<size_t>(slot) * TP_ROWS + row] =
              lt > 0.f ? (m + log2f(lt)) * 0.6931471805599453f : -INFINITY;
        // O / l goes out 16 columns at a time through this warp's 2 KB of
        // the (already consumed) exchange buffer: each lane writes its row,
        // then each store instruction covers two 64-byte row segments.
        if (!bad) {
          uint8_t* stg = reinterpret_cast<uint8_t*>(sm.xbuf[b]) + sw * 2048;
          const int rsub = lane >> 4, csub = lane & 15;
          float* dst0 = a.part_o + (static_cast<size_t>(slot) * TP_ROWS + 32 * qd + rsub) * 512 +
                        256 * rank + 128 * hh + csub;
          for (int c0 = 0; c0 < 128; c0 += 16) {
            float v[16];
            tmem_ld16(tmem + lane_base + TM_O + 128 * hh + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 4; ++u)
              *reinterpret_cast<float4*>(stg + lane * 64 + ((u ^ (lane & 3)) * 16)) =
                  make_float4(v[4 * u] * inv_l, v[4 * u + 1] * inv_l, v[4 * u + 2] * inv_l,
                              v[4 * u + 3] * inv_l);
            __syncwarp();
            // All loads before the stores: the compiler cannot prove that the
            // staging buffer and the output do not alias.
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
              const int rr = 2 * r + rsub;
              x[r] = *reinterpret_cast<const float*>(stg + rr * 64 + (((csub >> 2) ^ (rr & 3)) * 16) +
                                                     (csub & 3) * 4);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r)
              if (32 * qd + 2 * r + rsub < rows_valid)
                dst0[static_cast<size_t>(2 * r) * 512 + c0] = x[r];
            __syncwarp();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sm.o_empty);
          mbar_arrive_remote_relaxed(mapa_shared(smem_u32(&sm.x_sendok[b]), peer));  // the exchange buffer is free again
        }
      }
    }
    if (bad && lane == 0) note_timeout(sm, a.err);
  }
  tc_fence_before();
  __syncwarp();
  // The peer may still address this CTA's shared memory (st.async stores,
  // remote arrivals) until it reaches this barrier.
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool FP8>
size_t smem_bytes() { return sizeof(PairSmemT<FP8>) + 1024; }

template <bool FP8>
bool set_smem_attr() {
  static bool done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done[dev]) return true;
  if (cudaFuncSetAttribute(attend_tc_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes<FP8>())) != cudaSuccess)
    return false;
  if (dev >= 0 && dev < 64) done[dev] = true;
  return true;
}

// A [rows][576] matrix of 16-bit (bf16 or fp16) or 8-bit elements, boxes of
// box_cols x box_rows.
bool rows_map(TmapSpec* sp, const void* base, uint64_t rows, uint32_t box_cols, uint32_t box_rows,
              CUtensorMapSwizzle sw,
              CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  *sp = TmapSpec{};
  sp->dtype = dt;
  sp->rank = 2;
  sp->base = base;
  sp->dims[0] = 576;
  sp->dims[1] = rows;
  sp->strides[0] = 576 * (dt == CU_TENSOR_MAP_DATA_TYPE_UINT8 ? 1 : 2);
  sp->box[0] = box_cols;
  sp->box[1] = box_rows;
  sp->swizzle = sw;
  return true;
}

// A [rows][576] bf16 matrix seen as 3-D: (64 columns of a chunk, rows, the
// nine 64-column chunks). A box of (64, box_rows, n_chunks) lands in shared
// memory as n_chunks consecutive [box_rows][64] tiles with 128-byte swizzle,
// which is the layout of n_chunks separate 2-D boxes, in one TMA instruction.
bool chunks_map(TmapSpec* sp, const void* base, uint64_t rows, uint32_t box_rows,
                uint32_t n_chunks) {
  *sp = TmapSpec{};
  sp->dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  sp->rank = 3;
  sp->base = base;
  sp->dims[0] = 64;
  sp->dims[1] = rows;
  sp->dims[2] = 9;
  sp->strides[0] = 576 * 2;
  sp->strides[1] = 128;
  sp->box[0] = 64;
  sp->box[1] = box_rows;
  sp->box[2] = n_chunks;
  sp->swizzle = CU_TENSOR_MAP_SWIZZLE_128B;
  return true;
}

}  // namespace

bool attend_tc_supported(const Shape& s, mla_dtype dt) {
  return dt == MLA_BF16 && s.d_c == 512 && s.d_r == 64 && s.bs == TP_TOK;
}

// Number of CTA pairs that can be resident at once (the attention grid is
// that many clusters of two), or 0 if the kernel cannot be configured.
int attend_tc_max_pairs() {
  if (!set_smem_attr<false>() || !set_smem_attr<true>()) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(TP_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes<false>();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attend_tc_kernel<false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

namespace {

// Shared by the bf16 and fp8 launches: the kernel, its tensor maps, the
// pair grid of 2-CTA clusters and programmatic dependent launch.
template <bool FP8>
cudaError_t launch_pairs(const Shape& s, const void* cache, const float* row_scale,
                         int num_blocks, const int32_t* page_table, int max_blocks, int B,
                         int n_q, const Partition& p, const WsView& ws, const int32_t* seq_lens,
                         uint32_t* err, cudaStream_t st) {
  const uint64_t q_rows = static_cast<uint64_t>(B) * n_q * s.n_h;
  const uint64_t kv_rows = static_cast<uint64_t>(num_blocks) * TP_TOK;
  const CUtensorMapDataType qdt =
      FP8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  TmapSpec sp;
  CUtensorMap tqc, tqr, tkc, tkr;
  rows_map(&sp, ws.qabs, q_rows, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, qdt);
  if (!get_tmap(sp, &tqc)) return cudaErrorInvalidValue;
  rows_map(&sp, ws.qabs, q_rows, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B, qdt);
  if (!get_tmap(sp, &tqr)) return cudaErrorInvalidValue;
  bool chunked = false;
  if constexpr (FP8) {
    // e4m3 codes, unswizzled: a stage's 256 latent codes x 64 rows, and its
    // 32 rotary codes x 64 rows
    rows_map(&sp, cache, kv_rows, 256, 64, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_DATA_TYPE_UINT8);
    if (!get_tmap(sp, &tkc)) return cudaErrorInvalidValue;
    rows_map(&sp, cache, kv_rows, 32, 64, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_DATA_TYPE_UINT8);
    if (!get_tmap(sp, &tkr)) return cudaErrorInvalidValue;
  } else {
    // A stage's four latent boxes as one 3-D box; if the driver does not take
    // that view, four 2-D boxes.
    chunked = true;
    chunks_map(&sp, cache, kv_rows, 64, 4);
    if (!get_tmap(sp, &tkc)) chunked = false;
    if (!chunked) {
      rows_map(&sp, cache, kv_rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
      if (!get_tmap(sp, &tkc)) return cudaErrorInvalidValue;
    }
    rows_map(&sp, cache, kv_rows, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B);
    if (!get_tmap(sp, &tkr)) return cudaErrorInvalidValue;
  }
  if (!set_smem_attr<FP8>()) return cudaErrorInvalidValue;
  PairArgs a;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.tiles = ws.tiles;
  a.prefix = ws.prefix;
  a.bounds = ws.bounds;
  a.first_b = ws.first_b;
  a.part_o = ws.part_o;
  a.part_lse = ws.part_lse;
  a.qabs = static_cast<const uint16_t*>(ws.qabs);
  a.row_scale = row_scale;
  a.q_rows = static_cast<long long>(q_rows);
  a.chunked = chunked ? 1 : 0;
  a.err = err;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks;
  a.B = B;
  a.n_q = n_q;
  a.n_h = s.n_h;
  a.G = p.G;
  a.P = p.C;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.C, 1, 1);
  cfg.blockDim = dim3(kThreads<FP8>, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes<FP8>();
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the previous kernel finishes (the kernel waits for it
  // before reading anything)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, attend_tc_kernel<FP8>, tqc, tqr, tkc, tkr, a);
}

}  // namespace

cudaError_t launch_attend_tc(const Shape& s, const void* cache, int num_blocks,
                             const int32_t* page_table, int max_blocks, int B, int n_q,
                             const Partition& p, const WsView& ws, const int32_t* seq_lens,
                             uint32_t* err, cudaStream_t st) {
  return launch_pairs<false>(s, cache, nullptr, num_blocks, page_table, max_blocks, B, n_q, p, ws,
                             seq_lens, err, st);
}

cudaError_t launch_attend_tc_fp8(const Shape& s, const void* codes, const float* row_scale,
                                 int num_blocks, const int32_t* page_table, int max_blocks, int B,
                                 int n_q, const Partition& p, const WsView& ws,
                                 const int32_t* seq_lens, uint32_t* err, cudaStream_t st) {
  return launch_pairs<true>(s, codes, row_scale, num_blocks, page_table, max_blocks, B, n_q, p,
                            ws, seq_lens, err, st);
}

}  // namespace mla
