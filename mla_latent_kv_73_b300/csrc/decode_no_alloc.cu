// mla_decode_no_alloc: the decode call for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc, or any allocator, on the decode path.
// Examples are a serving loop that must never take the allocator's lock
// mid-step, an embedding runtime that owns every byte of device memory
// itself, and code running where an allocation failure must be impossible
// by construction. Such callers cannot provide mla_decode's workspace.
// This entry point takes no workspace. It uses one fixed array that lives
// in the library's device image instead: kNoAllocBytes of device memory on
// every GPU that loads the library, held until the process exits.
//
// Nothing in the array has to start at zero. Within one call, every byte
// of the workspace is written before it is read. Every call shares the one
// array per device, so calls whose GPU work overlaps (on different streams,
// or from several host threads) race on it. Callers must order them, for
// example by issuing them on one stream.
#include <cuda_runtime.h>

#include <mutex>

#include "mla_internal.h"

namespace {

constexpr size_t kNoAllocBytes = MLA_NO_ALLOC_WORKSPACE_BYTES;

static __device__ __align__(256) unsigned char g_no_alloc_ws[kNoAllocBytes];

constexpr int kMaxDevices = 64;
void* g_ws_ptr[kMaxDevices] = {};
std::mutex g_ws_mu;

// Device address of the array on the current device. The first call on a
// device looks it up; later calls reuse it for the life of the process (a
// cudaDeviceReset in between is not supported: the remembered address
// would belong to the destroyed context).
mla_status workspace_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_ws_mu);
  if (!g_ws_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_ws) != cudaSuccess || !p) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    g_ws_ptr[dev] = p;
  }
  *out = g_ws_ptr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_decode_no_alloc(const mla_config* cfg, mla_weights w, const void* q,
                                          const void* cache, int32_t num_blocks,
                                          const int32_t* page_table, int32_t max_blocks,
                                          const int32_t* seq_lens, int32_t B, int32_t n_q,
                                          float* out, cudaStream_t stream) {
  size_t need = 0;
  mla_status st = mla_decode_workspace_size(cfg, B, n_q, 0, &need);
  if (st != MLA_OK) return st;
  if (need > kNoAllocBytes) return MLA_ERR_WORKSPACE;  // request too large for the array
  void* ws = nullptr;
  st = workspace_address(&ws);
  if (st != MLA_OK) return st;
  return mla_decode(cfg, w, q, cache, num_blocks, page_table, max_blocks, seq_lens, B, n_q, out,
                    ws, kNoAllocBytes, stream);
}
