/*
 * mla.h: C ABI of libmla, the decode hot path of Multi-head Latent Attention
 * (MLA) over a paged latent KV cache, for NVIDIA B300 (sm_103a).
 *
 * What is computed. Each cached token keeps one row [c | k_rope] of
 * d_c + d_r elements, shared by all heads. Here c = x W_dkv and
 * k_rope = RoPE(x W_kr, pos). Sources: "Multi-head Latent Attention: the KV
 * cache, compressed", sections "The one formula" and "RoPE, and why the
 * explanations stop here"; "Multi-head Latent Attention and KV Cache
 * Compression", section "Caching one latent vector".
 *
 * A decode step for head h and query token i of sequence b computes
 *     q_lat  = W_uk[h] q_nope                      (absorbed query, d_c wide)
 *     q_pe   = RoPE(q_rope, pos_i)
 *     s_j    = (q_lat . c_j + q_pe . k_rope_j) * scale      for j <= pos_i
 *     p      = softmax(s)
 *     o_lat  = sum_j p_j c_j
 *     out    = o_lat W_uv[h]                       (d_v wide)
 * so no per-head key or value is ever materialised. Sources: "Multi-head
 * Latent Attention and KV Cache Compression", section "The absorption trick
 * and decoupled RoPE" (query- and value-side absorption); "Multi-head Latent
 * Attention: the KV cache, compressed", sections "Absorption: the part that
 * makes it free" and "RoPE, and why the explanations stop here" (the score
 * has a content part and a decoupled RoPE part).
 *
 * Conventions. All of these are readings where the pages are silent.
 *  - RoPE rotates the pair of dimensions (i, i + d_r/2) by the angle
 *    pos * rope_base^(-2i/d_r).
 *  - Positions are 0-based indices within a sequence. seq_lens[b] counts
 *    every cached token, including the n_q new ones. Query i therefore sits
 *    at pos_i = seq_lens[b] - n_q + i and attends to keys j <= pos_i.
 *  - Paged cache: token j of sequence b lives in row
 *    page_table[b * max_blocks + j / block_size] * block_size + j % block_size
 *    of the cache, viewed as [num_blocks * block_size, d_c + d_r].
 *  - The weights use the layouts below. Head h owns columns
 *    [h*d, (h+1)*d) of W_uk and W_uv.
 *
 * Memory and streams. Every pointer argument is a DEVICE pointer to memory
 * the caller owns and keeps alive until the work queued on `stream` has
 * finished. The only exception is the out-parameters of the host-side query
 * functions (mla_decode_workspace_size, mla_decode_full_workspace_size,
 * mla_decode_layer_workspace_size, mla_get_last_device_error), which are
 * host pointers. All compute calls are
 * asynchronous on `stream` and return once the work is queued. The library
 * allocates device memory only inside mla_absorb_weights and mla_fold_full.
 * It never allocates on the decode path.
 *
 * Errors. Each call checks its arguments on the host before queueing any
 * work. A failed check returns a status other than MLA_OK and queues
 * nothing. Problems that only the device can see (a page id out of range,
 * a sequence shorter than n_q, a wait that timed out) set bits in a
 * per-device error word. mla_get_last_device_error() reads and clears it.
 * Nothing in the library traps or aborts.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null pointer, negative count, bad enum */
  MLA_ERR_SHAPE = 2,         /* inconsistent or unsupported dimensions */
  MLA_ERR_CAPACITY = 3,      /* page table / cache too small for the request */
  MLA_ERR_UNSUPPORTED = 4,   /* valid request that this build or device cannot run */
  MLA_ERR_WORKSPACE = 5,     /* workspace missing, misaligned or too small */
  MLA_ERR_CUDA = 6,          /* a CUDA runtime call failed */
  MLA_ERR_DEVICE_CHECK = 7,  /* the device error word is non-zero */
  MLA_ERR_TIMEOUT = 8        /* a bounded device-side wait gave up */
} mla_status;

typedef enum { MLA_F32 = 0, MLA_BF16 = 1 } mla_dtype;

/* Which decode kernel to run. MLA_IMPL_AUTO picks the tensor-core kernel
 * when the shape and device allow it, and the CUDA-core kernel otherwise. */
typedef enum {
  MLA_IMPL_AUTO = 0,
  MLA_IMPL_CUDA_CORE = 1,    /* fp32 FMA kernel, any supported shape */
  MLA_IMPL_TENSOR_CORE = 2   /* tcgen05/TMEM kernel: bf16, d_c=512, d_r=64, block_size=64 */
} mla_impl;

/* Device error word bits (mla_get_last_device_error). */
#define MLA_DEVERR_PAGE_RANGE   0x1u  /* a page-table entry outside [0, num_blocks) */
#define MLA_DEVERR_SEQ_LEN      0x2u  /* seq_lens[b] < n_q or beyond the page table */
#define MLA_DEVERR_APPEND_INDEX 0x4u  /* append: seq_idx or pos outside the page table */
#define MLA_DEVERR_TIMEOUT      0x8u  /* a bounded mbarrier wait gave up */

typedef struct {
  int32_t n_h;            /* query heads */
  int32_t d_model;        /* hidden width (input of W_dkv, W_kr) */
  int32_t d_c;            /* latent width (cached) */
  int32_t d_r;            /* decoupled RoPE width (cached, shared by heads); even */
  int32_t d_nope;         /* per-head non-rotary query/key width */
  int32_t d_v;            /* per-head value width */
  int32_t block_size;     /* tokens per cache page */
  float rope_base;        /* RoPE base, e.g. 10000 */
  float softmax_scale;    /* 0 selects 1/sqrt(d_nope + d_r) */
  mla_dtype dtype;        /* dtype of cache, weights, x and q; outputs are fp32 */
  int32_t impl;           /* an mla_impl value */
} mla_config;
/* Supported shapes: n_h, d_model, d_nope, d_v, block_size >= 1; d_c a multiple
 * of 4 in [4, 512]; d_r even and >= 2; d_c + d_r <= 1024; d_nope <= 1024;
 * d_v <= 1024. Any other shape returns MLA_ERR_SHAPE before device work. */

typedef struct mla_weights_s* mla_weights; /* opaque, library-owned */

/* Fold the up-projections into the decode operands, once at load time.
 * Source: "Multi-head Latent Attention: the KV cache, compressed", section
 * "Store the archive, not the files" (build the fold once, at load);
 * "Multi-head Latent Attention and KV Cache Compression", section "The
 * absorption trick and decoupled RoPE" (W_uk goes to the query side and
 * W_uv to the output side).
 *   W_dkv [d_model, d_c], W_kr [d_model, d_r]       row-major, cfg->dtype
 *   W_uk  [d_c, n_h*d_nope], W_uv [d_c, n_h*d_v]   row-major, cfg->dtype
 * Allocates library-owned device buffers, runs the repacking kernels on
 * `stream` and waits for them, then returns the handle in *out. The packed
 * weights are complete and never written again while the handle lives, so
 * the decode kernels may load them before the previous kernel on their
 * stream has finished. The caller's weight buffers may be freed on return. Release the handle with
 * mla_weights_free. The handle is bound to the config it was built with and
 * to the current device. */
mla_status mla_absorb_weights(const mla_config* cfg, const void* W_dkv, const void* W_kr,
                              const void* W_uk, const void* W_uv, cudaStream_t stream,
                              mla_weights* out);

/* Free a handle from mla_absorb_weights. Waits for the device to finish
 * work that may still use it. NULL is accepted. */
mla_status mla_weights_free(mla_weights w);

/* Compress and append T new tokens to the paged latent cache.
 * Source: "Multi-head Latent Attention: the KV cache, compressed", sections
 * "The code" (latent) and "RoPE, and why the explanations stop here" (the
 * decoupled key is rotated and cached, one copy for all heads); "DeepSeek V3
 * Multi-Head Latent Attention (MLA): How It Slashes KV Cache Memory",
 * section "Low-Rank Key-Value Joint Compression".
 *   x          [T, d_model]               cfg->dtype
 *   seq_idx    [T] int32                  sequence of each token, in [0, B)
 *   pos        [T] int32                  position of each token in its sequence
 *   page_table [B, max_blocks] int32
 *   cache      [num_blocks, block_size, d_c + d_r] cfg->dtype, updated in place
 * Row t is written to the cache row given by the paged-layout convention.
 * Accumulation is fp32, and the result is rounded to nearest-even when
 * stored. Tokens whose seq_idx, pos or page id fall outside the tables are
 * skipped and set MLA_DEVERR_APPEND_INDEX or MLA_DEVERR_PAGE_RANGE. Two
 * tokens that name the same row race. T = 0 is a no-op. */
mla_status mla_append_kv(const mla_config* cfg, mla_weights w, const void* x,
                         const int32_t* seq_idx, const int32_t* pos, const int32_t* page_table,
                         int32_t B, int32_t max_blocks, void* cache, int32_t num_blocks,
                         int32_t T, cudaStream_t stream);

/* Bytes of device workspace that mla_decode needs for B sequences with n_q
 * query tokens each, on the current device. total_tokens (the sum of
 * seq_lens, or an upper bound; 0 if unknown) is accepted for interface
 * stability. The size does not depend on it. Writes the size to *bytes
 * (a host pointer). */
mla_status mla_decode_workspace_size(const mla_config* cfg, int32_t B, int32_t n_q,
                                     int64_t total_tokens, size_t* bytes);

/* Absorbed-query decode attention over the paged cache, with per-sequence
 * lengths. Steps a2..a5 in one call: absorb q, split-KV latent attention,
 * log-sum-exp combine, value up-projection.
 *   q          [B, n_q, n_h, d_nope + d_r] cfg->dtype, RoPE not yet applied
 *   cache      [num_blocks, block_size, d_c + d_r] cfg->dtype
 *   page_table [B, max_blocks] int32
 *   seq_lens   [B] int32, each in [n_q, max_blocks * block_size]
 *   out        [B, n_q, n_h, d_v] fp32
 *   workspace  device buffer of at least mla_decode_workspace_size() bytes,
 *              256-byte aligned. Its contents on entry do not matter.
 * Bad sequence lengths and page ids set the device error word. Their
 * outputs are then zero (bad lengths) or unspecified (bad pages). */
mla_status mla_decode(const mla_config* cfg, mla_weights w, const void* q, const void* cache,
                      int32_t num_blocks, const int32_t* page_table, int32_t max_blocks,
                      const int32_t* seq_lens, int32_t B, int32_t n_q, float* out,
                      void* workspace, size_t ws_bytes, cudaStream_t stream);

/* The three stages of mla_decode as separate calls, so that each kernel can
 * be timed on its own. Called in this order with the same arguments and
 * workspace, they produce exactly what mla_decode produces. Intermediate
 * results live in the workspace, in a layout private to the library.
 *   mla_decode_absorb_q   a2: q_lat = W_uk[h] q_nope, q_pe = RoPE(q_rope);
 *                              also plans the split-KV partition.
 *   mla_decode_attend     a3: split-KV attention over the latent cache.
 *   mla_decode_combine    a4+a5: log-sum-exp combine of the splits, then
 *                              out = o_lat W_uv[h].
 * The tensor-core kernel reads the cache with TMA, which needs a 16-byte
 * aligned cache pointer. For a misaligned cache under MLA_IMPL_AUTO,
 * mla_decode falls back to the CUDA-core kernel. The stage calls have to
 * agree on one partition, so they return MLA_ERR_INVALID_ARG instead. */
mla_status mla_decode_absorb_q(const mla_config* cfg, mla_weights w, const void* q,
                               const int32_t* seq_lens, int32_t max_blocks, int32_t B,
                               int32_t n_q, void* workspace, size_t ws_bytes,
                               cudaStream_t stream);
mla_status mla_decode_attend(const mla_config* cfg, const void* cache, int32_t num_blocks,
                             const int32_t* page_table, int32_t max_blocks,
                             const int32_t* seq_lens, int32_t B, int32_t n_q, void* workspace,
                             size_t ws_bytes, cudaStream_t stream);
mla_status mla_decode_combine(const mla_config* cfg, mla_weights w, const int32_t* seq_lens,
                              int32_t B, int32_t n_q, float* out, void* workspace,
                              size_t ws_bytes, cudaStream_t stream);

/* The attention core alone (a3 + a4): split-KV attention of queries that
 * are already in latent space over the paged cache, and the log-sum-exp
 * merge of the splits, with neither the W_uk fold nor the W_uv
 * up-projection.
 * Source: "Multi-head Latent Attention and KV Cache Compression", section
 * "The absorption trick and decoupled RoPE" (score = q_lat . c + q_pe .
 * k_rope; the output side keeps the weighted latent sum); "Multi-head
 * Latent Attention: the KV cache, compressed", section "RoPE, and why the
 * explanations stop here" (the position part is a separate product).
 *   q_abs      [B, n_q, n_h, d_c + d_r] cfg->dtype: per head [q_lat | q_pe],
 *              q_lat = W_uk[h]^T q_nope and q_pe = RoPE(q_rope, position)
 *              already applied, not yet scaled
 *   cache, page_table, seq_lens: as for mla_decode
 *   o_lat      [B, n_q, n_h, d_c] fp32: sum_j p_j c_j, p = softmax over the
 *              keys the query sees of scale * (q_lat . c_j + q_pe . k_rope_j);
 *              16-byte aligned (MLA_ERR_INVALID_ARG otherwise, before any
 *              work is queued)
 *   workspace  at least mla_decode_workspace_size() bytes, 256-byte aligned
 * The queries are copied into the workspace (times scale, in the attention
 * kernel's operand type), so q_abs has no alignment requirement. Errors as
 * for mla_decode. Needs no weights handle. */
mla_status mla_decode_latent(const mla_config* cfg, const void* q_abs, const void* cache,
                             int32_t num_blocks, const int32_t* page_table, int32_t max_blocks,
                             const int32_t* seq_lens, int32_t B, int32_t n_q, float* o_lat,
                             void* workspace, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * fp8 latent cache: e4m3 codes with one fp32 scale per cache row.
 *
 * Source: "Multi-head Latent Attention and KV Cache Compression", section
 * "Moving a trained MHA model over": quantisation can be stacked on the
 * latent cache, and its error passes through the up-projections into every
 * head. The page fixes neither the format nor the scale granularity. This
 * library takes e4m3 in the "fn" variant (bias 7, 3 mantissa bits, largest
 * finite value 448, no infinities) and one scale per row:
 *     scale = max_k |row[k]| / 448   (1 for a row of zeros)
 *     code[k] = e4m3(row[k] / scale), round to nearest, ties to even,
 *               saturating at +-448
 * with the scale and the division in fp32. A row dequantises to
 * code[k] * scale. The cache layouts:
 *   cache      [num_blocks, block_size, d_c + d_r] uint8 (e4m3 codes)
 *   row_scale  [num_blocks, block_size] fp32
 * Half the bytes of a bf16 cache per token, plus 4 bytes of scale.
 * These calls need a bf16 config with d_c = 512, d_r = 64, d_nope = d_v =
 * 128 and 64-token blocks (the tensor-core kernels), else they return
 * MLA_ERR_UNSUPPORTED. Pointers to cache, row_scale, q and x must be 16-byte
 * aligned (MLA_ERR_INVALID_ARG otherwise).
 * ------------------------------------------------------------------------ */

/* Quantise T fp32 rows and place them in the fp8 cache.
 *   rows       [T, d_c + d_r] fp32 (device), row t belongs to token t
 *   seq_idx, pos, page_table, B, max_blocks: as for mla_append_kv
 * Writes each row's codes and scale to the cache row that the paged layout
 * gives. Bad indices are skipped and set MLA_DEVERR_APPEND_INDEX or
 * MLA_DEVERR_PAGE_RANGE. T = 0 is a no-op. */
mla_status mla_quantize_rows_fp8(const mla_config* cfg, const float* rows, const int32_t* seq_idx,
                                 const int32_t* pos, const int32_t* page_table, int32_t B,
                                 int32_t max_blocks, void* cache, float* row_scale,
                                 int32_t num_blocks, int32_t T, cudaStream_t stream);

/* Bytes of device workspace that mla_append_kv_fp8 needs for T tokens: the
 * fp32 rows of up to 256 tokens at a time. Writes the size to *bytes. */
mla_status mla_append_kv_fp8_workspace_size(const mla_config* cfg, int32_t T, size_t* bytes);

/* mla_append_kv into an fp8 cache: the rows [x W_dkv | RoPE(x W_kr, pos)]
 * are computed in fp32 (256 tokens at a time, into the workspace), then
 * quantised and placed as by mla_quantize_rows_fp8. Arguments as for
 * mla_append_kv; workspace: at least mla_append_kv_fp8_workspace_size()
 * bytes, 256-byte aligned, contents on entry irrelevant. */
mla_status mla_append_kv_fp8(const mla_config* cfg, mla_weights w, const void* x,
                             const int32_t* seq_idx, const int32_t* pos,
                             const int32_t* page_table, int32_t B, int32_t max_blocks,
                             void* cache, float* row_scale, int32_t num_blocks, int32_t T,
                             void* workspace, size_t ws_bytes, cudaStream_t stream);

/* mla_decode over an fp8 cache: the same absorbed-query attention on the
 * dequantised rows (code * scale), with the same workspace
 * (mla_decode_workspace_size). The queries are absorbed into fp16, the
 * cache codes are widened to fp16 (exact) inside the attention kernel, the
 * MMAs accumulate in fp32, and each row's scale multiplies its score and
 * its value weight. Bad lengths and page ids behave as for mla_decode. */
mla_status mla_decode_fp8(const mla_config* cfg, mla_weights w, const void* q, const void* cache,
                          const float* row_scale, int32_t num_blocks, const int32_t* page_table,
                          int32_t max_blocks, const int32_t* seq_lens, int32_t B, int32_t n_q,
                          float* out, void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Size of the fixed device array that mla_decode_no_alloc uses in place of a
 * workspace: 32 MiB. */
#define MLA_NO_ALLOC_WORKSPACE_BYTES ((size_t)32 << 20)

/* mla_decode for callers that cannot allocate device memory. The paper has
 * no counterpart to this call: it is a deployment convenience.
 * Some callers are not allowed to call cudaMalloc or any other allocator on
 * the decode path. Examples are a serving loop that must not take an
 * allocator lock mid-step, and a runtime that hands out all device memory
 * itself. Such callers cannot supply mla_decode's workspace. This call takes
 * the same arguments as mla_decode minus the workspace, and computes the same
 * result. Its scratch space is one array of MLA_NO_ALLOC_WORKSPACE_BYTES
 * inside the library's device image, which every GPU that loads the library
 * holds until the process exits. The call allocates nothing.
 *  - Returns MLA_ERR_WORKSPACE, and queues nothing, when the request needs
 *    more scratch than the array holds (see mla_decode_workspace_size).
 *  - The first call on each device looks up the array's device address.
 *    Make that first call before any stream capture.
 *  - All calls on a device share the array. It keeps the previous call's
 *    contents, and nothing in it needs to start at zero. Calls whose GPU work
 *    overlaps (other streams, other host threads) race on it, so order them,
 *    for example by issuing them on one stream.
 *  - The array's address is remembered per device for the life of the
 *    process. Resetting a device (cudaDeviceReset) after the first call is
 *    not supported: later calls on that device would use a stale address.
 *  - On a B300 the DeepSeek-V2 shape (128 heads) fits with batch 16 (24.8
 *    MiB) or batch 4 with 2 query tokens (21.7 MiB); batch 64 needs 43.6 MiB
 *    and is rejected. The workspace does not depend on the cached lengths. */
mla_status mla_decode_no_alloc(const mla_config* cfg, mla_weights w, const void* q,
                               const void* cache, int32_t num_blocks, const int32_t* page_table,
                               int32_t max_blocks, const int32_t* seq_lens, int32_t B,
                               int32_t n_q, float* out, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Full-fold variant: one attention layer from the hidden state.
 *
 * Both up-projections are folded into the neighbouring projections once,
 * at load, so the decode call takes the query token's hidden state x_q and
 * returns the layer output y:
 *     W_abs[h] = W_q,nope[h] W_uk[h]^T      (d_model x d_c)
 *     W_vo[h]  = W_uv[h] W_o[h]             (d_c x d_model)
 *     q_lat    = x_q W_abs[h],  q_pe = RoPE(x_q W_qr[h], pos_i)
 *     o_lat    = the latent attention of mla_decode
 *     y        = sum_h o_lat[h] W_vo[h]  =  concat_h(o_h) W_o
 * Sources: "Multi-head Latent Attention: the KV cache, compressed", sections
 * "Store the archive, not the files" (fold W_q and W_uk once, at load) and
 * "The code" (absorb_q_into_latent; decoupled_score keeps the rotary query
 * block W_qr out of the fold); "Multi-head Latent Attention and KV Cache
 * Compression", section "The absorption trick and decoupled RoPE" (W_uv
 * folds into the output projection).
 * The first page's caveat applies: at DeepSeek-V2 widths the folded
 * matrices are far larger than W_uk and W_uv (4.5x on the query side and
 * 40x on the output side), so this form pays only at small widths. The
 * per-head path above is the one for large models.
 * ------------------------------------------------------------------------ */
typedef struct mla_full_weights_s* mla_full_weights; /* opaque, library-owned */

/* Build the folded matrices, once at load.
 *   W_q  [d_model, n_h*(d_nope + d_r)] row-major, cfg->dtype; head h owns
 *        columns [h*(d_nope+d_r), (h+1)*(d_nope+d_r)) as [q_nope | q_rope]
 *   W_uk [d_c, n_h*d_nope], W_uv [d_c, n_h*d_v]  as in mla_absorb_weights
 *   W_o  [n_h*d_v, d_model] row-major, cfg->dtype; head h's output meets
 *        rows [h*d_v, (h+1)*d_v)
 * The folded matrices are stored in fp32, d_model*n_h*(d_c+d_r) +
 * n_h*d_c*d_model elements; the fold accumulates in fp64. Allocates them,
 * queues the folding kernels on `stream` and returns the handle in *out.
 * The caller's buffers may be freed once `stream` has passed this call.
 * Release the handle with mla_full_weights_free. */
mla_status mla_fold_full(const mla_config* cfg, const void* W_q, const void* W_uk,
                         const void* W_uv, const void* W_o, cudaStream_t stream,
                         mla_full_weights* out);

/* Free a handle from mla_fold_full. Waits for the device to finish work
 * that may still use it. NULL is accepted. */
mla_status mla_full_weights_free(mla_full_weights w);

/* Bytes of device workspace that mla_decode_full needs for B sequences with
 * n_q query tokens each, on the current device. Writes the size to *bytes
 * (a host pointer). */
mla_status mla_decode_full_workspace_size(const mla_config* cfg, int32_t B, int32_t n_q,
                                          size_t* bytes);

/* The attention layer for B sequences with n_q new tokens each.
 *   x_q        [B, n_q, d_model] cfg->dtype: hidden states of the query tokens
 *   cache, num_blocks, page_table, max_blocks, seq_lens  as in mla_decode
 *   y          [B, n_q, d_model] fp32 layer output
 *   workspace  device buffer of at least mla_decode_full_workspace_size()
 *              bytes, 256-byte aligned; its contents on entry do not matter
 * The query projection and the output projection accumulate in fp32 (the
 * projected query is rounded to cfg->dtype before the attention, like q in
 * mla_decode). The decode kernel is chosen as in mla_decode. Errors as in
 * mla_decode. */
mla_status mla_decode_full(const mla_config* cfg, mla_full_weights fw, const void* x_q,
                           const void* cache, int32_t num_blocks, const int32_t* page_table,
                           int32_t max_blocks, const int32_t* seq_lens, int32_t B, int32_t n_q,
                           float* y, void* workspace, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * One layer's decode step: append, decode and the output projection.
 *
 * The per-head path leaves the output projection W_o with the caller. This
 * call runs the whole step of one attention layer for the new tokens on
 * `stream`: mla_append_kv of their hidden states, mla_decode of their
 * queries, then y = concat_h(o_h) W_o. The kernels are chained with
 * programmatic dependent launch: each one's constant-weight prologue overlaps
 * the kernel before it, and the projection streams W_o while the combine
 * still runs. Source for the projection's place in the layer: "Multi-head
 * Latent Attention: the KV cache, compressed", section "What it costs, said
 * plainly" (W_o [n_h*head_dim -> d_model] among the layer's weights).
 * ------------------------------------------------------------------------ */

/* Bytes of device workspace that mla_decode_layer needs (the decode's, the
 * bf16 hi/lo copy of out that the tensor-core projection reads for up to 64
 * new tokens, and the projection's split partials). Writes the size to
 * *bytes (a host pointer). */
mla_status mla_decode_layer_workspace_size(const mla_config* cfg, int32_t B, int32_t n_q,
                                           size_t* bytes);

/* One decode step of one layer for B sequences with n_q new tokens each.
 *   W_o        [n_h*d_v, d_model] row-major, cfg->dtype, caller-owned; head
 *              h's output meets rows [h*d_v, (h+1)*d_v)
 *   x          [B*n_q, d_model] cfg->dtype: hidden states of the new tokens
 *   seq_idx, pos [B*n_q] int32: their sequences and positions (as in
 *              mla_append_kv; normally pos = seq_lens[b] - n_q + i)
 *   q          [B, n_q, n_h, d_nope + d_r] cfg->dtype, RoPE not yet applied
 *   cache      updated in place with the new rows, then read
 *   out        [B, n_q, n_h, d_v] fp32: the per-head outputs (also returned)
 *   y          [B, n_q, d_model] fp32: the layer output
 *   workspace  at least mla_decode_layer_workspace_size() bytes, 256-byte
 *              aligned
 * The projection accumulates in fp32. With the tensor-core decode, up to 64
 * new tokens, d_model and n_h*d_v multiples of 8, a 16-byte aligned W_o and
 * a 16-byte aligned out, it runs on the tensor cores: out enters as a bf16
 * hi + lo pair (about 16 bits of its mantissa). Otherwise it runs on the
 * CUDA cores from out in fp32. Errors as in mla_append_kv and mla_decode. */
mla_status mla_decode_layer(const mla_config* cfg, mla_weights w, const void* W_o, const void* x,
                            const int32_t* seq_idx, const int32_t* pos, const void* q,
                            void* cache, int32_t num_blocks, const int32_t* page_table,
                            int32_t max_blocks, const int32_t* seq_lens, int32_t B, int32_t n_q,
                            float* out, float* y, void* workspace, size_t ws_bytes,
                            cudaStream_t stream);

/* Which decode kernel mla_decode would run for this config on the current
 * device. Writes an mla_impl value other than MLA_IMPL_AUTO to *impl, a host
 * pointer. */
mla_status mla_decode_impl(const mla_config* cfg, int32_t* impl);

/* Synchronise `stream`, then read and clear the current device's error word
 * into *code (a host pointer). Returns MLA_ERR_DEVICE_CHECK if the word was
 * non-zero. */
mla_status mla_get_last_device_error(cudaStream_t stream, uint32_t* code);

/* Static, human-readable name of a status code. */
const char* mla_status_string(mla_status s);

#ifdef __cplusplus
}
#endif
#endif /* MLA_H_ */
