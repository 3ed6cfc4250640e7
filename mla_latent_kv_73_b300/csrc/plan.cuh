// Split-KV plan, written by one CTA of the query-absorption kernel: the
// number of 64-token tiles of each sequence and their exclusive prefix sum.
// The attention and combine kernels read both. A sequence whose length is
// below n_q or beyond its page table gets 0 tiles and sets MLA_DEVERR_SEQ_LEN.
#pragma once
#include "device_common.cuh"

namespace mla {

// Every thread of the block (NT threads) must call this.
template <int NT>
__device__ void write_plan(const int32_t* __restrict__ seq_lens, int B, int n_q, int max_blocks,
                           int bs, int TS, int32_t* tiles, int32_t* prefix, uint32_t* err) {
  __shared__ int32_t warp_sums[NT / 32];
  __shared__ int32_t carry;
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
    if (b < B) prefix[b] = before + v - t;
    __syncthreads();
    if (threadIdx.x == NT - 1) carry = before + v;
    __syncthreads();
  }
  if (threadIdx.x == 0) prefix[B] = carry;
}


}  // namespace mla
