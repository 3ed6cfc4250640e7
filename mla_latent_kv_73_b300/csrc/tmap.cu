// Tensor-map encoding through the driver entry point, with a cache keyed by
// the full description of the map.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "tmap.h"

namespace mla {
namespace {

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

bool same(const TmapSpec& a, const TmapSpec& b) { return std::memcmp(&a, &b, sizeof(a)) == 0; }

struct Cache {
  static constexpr int kSlots = 64;
  struct Entry {
    bool used = false;
    TmapSpec spec;
    CUtensorMap map;
  } e[kSlots];
  int next = 0;
  std::mutex mu;
};

}  // namespace

bool get_tmap(const TmapSpec& in, CUtensorMap* out) {
  TmapSpec spec;
  std::memset(&spec, 0, sizeof(spec));  // padding bytes take part in the key
  spec.dtype = in.dtype;
  spec.rank = in.rank;
  spec.base = in.base;
  for (int i = 0; i < in.rank; ++i) {
    spec.dims[i] = in.dims[i];
    spec.box[i] = in.box[i];
    if (i + 1 < in.rank) spec.strides[i] = in.strides[i];
  }
  spec.swizzle = in.swizzle;
  static Cache cache;
  std::lock_guard<std::mutex> lk(cache.mu);
  for (auto& x : cache.e) {
    if (x.used && same(x.spec, spec)) {
      *out = x.map;
      return true;
    }
  }
  auto fn = encode_fn();
  if (!fn || spec.rank < 1 || spec.rank > 5) return false;
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5], es[5];
  for (int i = 0; i < spec.rank; ++i) {
    dims[i] = spec.dims[i];
    box[i] = spec.box[i];
    es[i] = 1;
    if (i + 1 < spec.rank) strides[i] = spec.strides[i];
  }
  CUtensorMap m;
  if (fn(&m, spec.dtype, spec.rank, const_cast<void*>(spec.base), dims, strides, box, es,
         CU_TENSOR_MAP_INTERLEAVE_NONE, spec.swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  auto& slot = cache.e[cache.next];
  cache.next = (cache.next + 1) % Cache::kSlots;
  slot.used = true;
  slot.spec = spec;
  slot.map = m;
  *out = m;
  return true;
}

}  // namespace mla
