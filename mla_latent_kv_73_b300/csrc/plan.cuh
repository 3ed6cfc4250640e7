// Split-KV plan, written by one CTA of the query-absorption kernel: the
// number of 64-token tiles of each sequence, their exclusive prefix sum, and
// the first work item of each of the C ranges. The attention and combine
// kernels read all three. A sequence whose length is below n_q or beyond its
// page table gets 0 tiles and sets MLA_DEVERR_SEQ_LEN.
//
// Range boundaries. Work items are (g, b, tile) in group-major order. Each
// range is charged its tiles plus K for every (g, b) piece it contains; the
// cumulative cost up to item (g, b, j) is taken as
//   F(g, b, j) = g T + prefix[b] + j + K (g B + b)
// (T tiles in all, one K per sequence start) and range c begins at the first
// item whose F reaches c F_total / C. F is monotone in the item, so each
// boundary is an independent binary search; with K = 0 the ranges have equal
// length. first_b[c] is the sequence of range c's first item (0 for an empty
// range), so the attention kernel finds its first piece without a search.
#pragma once
#include "device_common.cuh"

namespace mla {

// Sequences whose tiles and prefix sums the plan writer also keeps in shared
// memory, so that its boundary searches are shared-memory reads rather than
// dependent round trips to L2.
constexpr int PLAN_SMEM_B = 1024;

// Every thread of the block (NT threads) must call this.
template <int NT>
__device__ void write_plan(const int32_t* __restrict__ seq_lens, int B, int n_q, int max_blocks,
                           int bs, int TS, int G, int C, int K, int32_t* tiles, int32_t* prefix,
                           long long* bounds, int32_t* first_b, uint32_t* err) {
  __shared__ int32_t warp_sums[NT / 32];
  __shared__ int32_t carry;
  __shared__ int32_t s_tiles[PLAN_SMEM_B], s_prefix[PLAN_SMEM_B + 1];
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  for (int b0 = 0; b0 < B; b0 += NT) {
    const int b = b0 + threadIdx.x;
    int t = 0;
    if (b < B) {
      const long long L = seq_lens[b];
      if (L < n_q || L > static_cast<long long>(max_blocks) * bs) {
        set_error(err, MLA_DEVERR_SEQ_LEN);
      } else {
        t = static_cast<int>((L + TS - 1) / TS);
      }
      tiles[b] = t;
      if (b < PLAN_SMEM_B) s_tiles[b] = t;
    }
    // inclusive warp scan
    int v = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    int before = carry;
    for (int w = 0; w < warp; ++w) before += warp_sums[w];
    if (b < B) {
      prefix[b] = before + v - t;
      if (b < PLAN_SMEM_B) s_prefix[b] = before + v - t;
    }
    __syncthreads();
    if (threadIdx.x == NT - 1) carry = before + v;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    prefix[B] = carry;
    if (B <= PLAN_SMEM_B) s_prefix[B] = carry;
  }
  __syncthreads();  // tiles and prefix are visible to the whole block
  const bool in_smem = B <= PLAN_SMEM_B;
  const int32_t* P = in_smem ? s_prefix : prefix;
  const int32_t* TL = in_smem ? s_tiles : tiles;
  const long long T = carry;
  const long long per_g = T + static_cast<long long>(K) * B;  // F of one whole group
  const long long F_total = per_g * G;
  for (int c = threadIdx.x; c <= C; c += NT) {
    long long v = 0;
    if (c == C) {
      v = T * G;
    } else if (c > 0 && F_total > 0) {
      const long long Fc = (static_cast<long long>(c) * F_total) / C;
      const int g = static_cast<int>(min(static_cast<long long>(G - 1), Fc / per_g));
      const long long r = Fc - g * per_g;
      int lo = 0, hi = B;  // largest b with prefix[b] + K b <= r
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (P[mid] + static_cast<long long>(K) * mid <= r) lo = mid; else hi = mid;
      }
      // past the end of sequence lo: cut at its end (the next sequence's start)
      const long long j = min(r - P[lo] - static_cast<long long>(K) * lo,
                              static_cast<long long>(TL[lo]));
      v = g * T + P[lo] + j;
    }
    bounds[c] = v;
    if (c < C) {
      int b = 0;
      if (T > 0 && v < T * G) {
        const long long rem = v % T;
        int lo = 0, hi = B;  // largest b with prefix[b] <= rem: the sequence holding item v
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (P[mid] <= rem) lo = mid; else hi = mid;
        }
        b = lo;
      }
      first_b[c] = b;
    }
  }
}

// The range holding work item x: the largest c < C with rb[c] <= x, for
// boundaries rb[0..C] and 0 <= x < rb[C]. Empty ranges are never returned.
__device__ __forceinline__ int range_of_item(const long long* rb, int C, long long x) {
  int lo = 0, hi = C;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (rb[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}


}  // namespace mla
