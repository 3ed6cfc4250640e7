// Internal declarations shared by the libmla translation units.
#pragma once
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/mla.h"

namespace mla {

// Shape as the kernels see it.
struct Shape {
  int n_h, d_model, d_c, d_r, d_nope, d_v, bs;
  float rope_base, scale;
#ifdef __CUDACC__
  __host__ __device__
#endif
  int R() const { return d_c + d_r; }
};

// Split-KV partition of one decode call.
//
// The query rows of a sequence, r = i*n_h + h for query token i and head h,
// are cut into G groups of RG rows. The cached tokens of sequence b form
// tiles_b = ceil(L_b / TS) tiles. The attention grid splits the flat list of
// work items (g, b, tile), ordered group-major, into C contiguous ranges:
// one per CTA (CUDA-core kernel) or per 2-CTA cluster (tensor-core kernel).
// A range costs its tiles plus K tiles for every (g, b) piece it starts
// (the partial's epilogue and the next piece's query load), and the plan
// writer cuts the item list so that these costs come out near-equal (K = 0
// gives ranges of equal length). One range therefore covers pieces of several
// (g, b) pairs. The piece of range c on pair (g, b) writes its partial result
// to slot c + g*B + b. The slots are unique, and slots = C + G*B bound their
// number.
struct Partition {
  int RG, G, TS, C, K, slots;
};

// Pointers into the decode workspace.
struct WsView {
  void* qabs;         // [B*n_q*n_h, R] in the cache dtype: [q_lat | RoPE(q_rope)]
  int32_t* tiles;     // [B]    tiles per sequence (0 for an invalid length)
  int32_t* prefix;    // [B+1]  exclusive prefix sum of tiles
  long long* bounds;  // [C+1]  first work item of each range (bounds[C] = all items)
  int32_t* first_b;   // [C]    sequence of each range's first work item
  float* part_o;      // [slots, RG, d_c] normalised partial latent outputs
  float* part_lse;    // [slots, RG]      natural-log sum-exp of each partial
};

struct WsLayout {
  size_t qabs, tiles, prefix, bounds, first_b, part_o, part_lse, total;
};

// q_bytes: bytes per stored query element (4 for the CUDA-core attention,
// the cache dtype's size for the tensor-core one).
WsLayout ws_layout(const Shape& s, int q_bytes, int B, int n_q, const Partition& p);
WsView ws_view(void* base, const WsLayout& l);

// Library-owned packed weights.
struct Weights {
  Shape shape;
  mla_dtype dtype;
  int device;
  void* w_dkvr;   // [R][d_model]: column j of [W_dkv | W_kr] stored contiguously.
                  // The d_r rotary columns are interleaved so that rotary
                  // dims i and i + d_r/2 sit in adjacent packed columns.
  void* w_uk;     // [n_h][d_c][d_nope]
  void* w_uv;     // [n_h][d_v][d_c]: per head, one contiguous d_c row per output
  uint64_t* rope_turns;  // [d_r/2] rope_base^(-2i/d_r) / (2 pi) as a 64-bit fraction of a turn
};

// Library-owned weights of the full-fold variant (x_q in, y out).
struct FullWeights {
  Shape shape;
  mla_dtype dtype;
  int device;
  float* w_qf;       // [d_model][n_h*R]: per head [W_abs[h] | W_qr[h]] (fp32)
  float* w_vo;       // [n_h*d_c][d_model]: row h*d_c + c of W_uv[h] W_o[h] (fp32)
  uint64_t* rope_turns;  // [d_r/2] rope_base^(-2i/d_r) / (2 pi) as a 64-bit fraction of a turn
};

// Split of K across CTAs for one x W product: S splits of k_split each.
struct XwPlan {
  int S, k_split;
};

// ---------------------------------------------------------------- launchers
// Each returns the cudaError_t of its launch.
cudaError_t launch_pack_weights(const Shape& s, mla_dtype dt, const void* W_dkv, const void* W_kr,
                                const void* W_uk, const void* W_uv, Weights* w, cudaStream_t st);

cudaError_t launch_append(const Shape& s, mla_dtype dt, const Weights* w, const void* x,
                          const int32_t* seq_idx, const int32_t* pos, const int32_t* page_table,
                          int B, int max_blocks, void* cache, int num_blocks, int T,
                          uint32_t* err, cudaStream_t st);
// The append's rows [x W_dkv | RoPE(x W_kr, pos)] in fp32, dense ([T][R], row
// t for token t), for the fp8 quantiser; nothing is written to a cache.
cudaError_t launch_append_rows_f32(const Shape& s, mla_dtype dt, const Weights* w, const void* x,
                                   const int32_t* seq_idx, const int32_t* pos, int T,
                                   float* rows, uint32_t* err, cudaStream_t st);

// fp8 (e4m3) latent cache: dense fp32 rows -> one scale per row and e4m3
// codes, placed through the page table (fp8.cu).
cudaError_t launch_quantize_rows_fp8(const Shape& s, const float* rows, const int32_t* seq_idx,
                                     const int32_t* pos, const int32_t* page_table, int B,
                                     int max_blocks, uint8_t* codes, float* row_scale,
                                     int num_blocks, int T, uint32_t* err, cudaStream_t st);

// out_scale multiplies q_lat and q_pe before they are stored (the
// tensor-core attention folds scale * log2(e) in here). q_f32: store them in
// fp32 (the CUDA-core attention's queries), else in the cache dtype.
cudaError_t launch_absorb_q(const Shape& s, mla_dtype dt, const Weights* w, const void* q,
                            const int32_t* seq_lens, int max_blocks, int B, int n_q,
                            const Partition& p, const WsView& ws, float out_scale, bool q_f32,
                            uint32_t* err, cudaStream_t st);

cudaError_t launch_attend_simt(const Shape& s, mla_dtype dt, const void* cache, int num_blocks,
                               const int32_t* page_table, int max_blocks, int B, int n_q,
                               const Partition& p, const WsView& ws, const int32_t* seq_lens,
                               uint32_t* err, cudaStream_t st);

// Tensor-core attention (bf16, d_c = 512, d_r = 64, block_size = 64), one
// 2-CTA cluster per work range; attend_tc_max_pairs() is how many clusters
// fit on the current device at once (0 if none).
bool attend_tc_supported(const Shape& s, mla_dtype dt);
int attend_tc_max_pairs();
cudaError_t launch_attend_tc(const Shape& s, const void* cache, int num_blocks,
                             const int32_t* page_table, int max_blocks, int B, int n_q,
                             const Partition& p, const WsView& ws, const int32_t* seq_lens,
                             uint32_t* err, cudaStream_t st);
// The same over an fp8 (e4m3) cache with one fp32 scale per row
// (row_scale[num_blocks * 64]); the queries in the workspace are fp16.
cudaError_t launch_attend_tc_fp8(const Shape& s, const void* codes, const float* row_scale,
                                 int num_blocks, const int32_t* page_table, int max_blocks, int B,
                                 int n_q, const Partition& p, const WsView& ws,
                                 const int32_t* seq_lens, uint32_t* err, cudaStream_t st);

// Tensor-core absorption and combine (bf16, d_c = 512, d_nope = 128, d_r = 64,
// d_v = 128). The query pointer must be 16-byte aligned for the TMA.
// q_half: store the absorbed queries in fp16 (for the attention over an fp8
// cache) instead of bf16.
bool absorb_tc_supported(const Shape& s, mla_dtype dt);
cudaError_t launch_absorb_q_tc(const Shape& s, const Weights* w, const void* q,
                               const int32_t* seq_lens, int max_blocks, int B, int n_q,
                               const Partition& p, const WsView& ws, float out_scale,
                               bool q_half, uint32_t* err, cudaStream_t st);
// hilo (optional, else null): out also as bf16 hi [B*n_q][n_h*d_v] followed
// by bf16 lo = bf16(out - hi), the operand of launch_proj_tc.
bool combine_tc_supported(const Shape& s, mla_dtype dt);
cudaError_t launch_combine_tc(const Shape& s, const Weights* w, int B, int n_q,
                              const Partition& p, const WsView& ws, float* out, uint16_t* hilo,
                              uint32_t* err, cudaStream_t st);

// The merge alone on the tensor-core partition (d_c = 512): o_lat
// [B*n_q][n_h][512] fp32, without the up-projection.
bool combine_latent_tc_supported(const Shape& s);
cudaError_t launch_combine_latent_tc(const Shape& s, int B, int n_q, const Partition& p,
                                     const WsView& ws, float* olat, uint32_t* err,
                                     cudaStream_t st);

cudaError_t launch_combine(const Shape& s, mla_dtype dt, const Weights* w,
                           const int32_t* seq_lens, int B, int n_q, const Partition& p,
                           const WsView& ws, float* out, cudaStream_t st);

// Full-fold variant and output projection. launch_fold_full builds
// FullWeights' matrices from the caller's W_q, W_uk, W_uv and W_o (all in
// dt). launch_xw computes out[M][N] = A[M][K] W[K][N] (A in a_dt, W in w_dt,
// out fp32) with the split-K plan from xw_plan; part holds xw_part_floats()
// floats of split partials; pdl launches it with programmatic dependent
// launch (its W stream may overlap the previous kernel).
// launch_q_finish turns the fp32 query projection [B*n_q][n_h*R] into the
// workspace's qabs (RoPE on the rotary block, times out_scale, rounded to
// dt) and writes the split-KV plan. launch_combine_latent merges the splits
// into o_lat [B*n_q][n_h*d_c] fp32 without the W_uv up-projection.
cudaError_t launch_fold_full(const Shape& s, mla_dtype dt, const void* W_q, const void* W_uk,
                             const void* W_uv, const void* W_o, FullWeights* w, int sms,
                             cudaStream_t st);
XwPlan xw_plan(int M, int K, int N, int sms);
size_t xw_part_floats(int M, int N, const XwPlan& p);
cudaError_t launch_xw(mla_dtype a_dt, const void* A, int M, int K, mla_dtype w_dt,
                      const void* W, int N, float* out, float* part, const XwPlan& p,
                      uint32_t* err, bool pdl, cudaStream_t st);
cudaError_t launch_q_finish(const Shape& s, mla_dtype dt, const uint64_t* rope_turns,
                            const float* qpre, const int32_t* seq_lens, int max_blocks, int B,
                            int n_q, const Partition& p, const WsView& ws, float out_scale,
                            bool q_f32, uint32_t* err, cudaStream_t st);
cudaError_t launch_combine_latent(const Shape& s, int B, int n_q, const Partition& p,
                                  const WsView& ws, float* olat, cudaStream_t st);
// The workspace's qabs = out_scale * q_abs (caller-absorbed queries in dt;
// fp32 when q_f32, else dt) and the split-KV plan, for mla_decode_latent.
cudaError_t launch_latent_q(const Shape& s, mla_dtype dt, const void* q_abs,
                            const int32_t* seq_lens, int max_blocks, int B, int n_q,
                            const Partition& p, const WsView& ws, float out_scale, bool q_f32,
                            uint32_t* err, cudaStream_t st);
// out[i] = sum_z part[z][i] over the S splits, in increasing z.
cudaError_t launch_sum_splits(const float* part, int S, size_t n, float* out, cudaStream_t st);

// Tensor-core output projection y[M x N] = A W for up to PROJ_TC_MAX_TOKENS
// rows of A, given as bf16 hi [M][K] followed by bf16 lo [M][K] (A = hi +
// lo), and W [K][N] bf16 row-major. proj_tc_applies: the sizes and W's
// alignment suit the kernel. proj_tc_plan: the K split (part needs S*M*N
// floats when S > 1).
constexpr int PROJ_TC_MAX_TOKENS = 64;
bool proj_tc_applies(int M, int K, int N, const void* W);
XwPlan proj_tc_plan(int M, int K, int N, int sms);
cudaError_t launch_proj_tc(const uint16_t* hilo, int M, int K, const void* W, int N, float* y,
                           float* part, const XwPlan& p, uint32_t* err, cudaStream_t st);

// Partition parameters for each attention kernel.
// tc_pairs: CTA pairs resident at once for the tensor-core attention kernel.
Partition partition_for(int impl, const Shape& s, int B, int n_q, int num_sms, int tc_pairs);

}  // namespace mla
