// Host helpers for TMA tensor maps: the driver's encoder, looked up once
// through the runtime, and a small cache of encoded maps. A map depends only
// on its base address, shape, strides, box and swizzle, so repeated decode
// calls on the same buffers reuse it instead of encoding it again.
#pragma once
#include <cuda.h>

#include <cstdint>

namespace mla {

struct TmapSpec {
  CUtensorMapDataType dtype;
  int rank;                 // 1..5
  const void* base;
  uint64_t dims[5];         // innermost first, in elements
  uint64_t strides[4];      // bytes, of dims 1..rank-1
  uint32_t box[5];          // elements per dimension
  CUtensorMapSwizzle swizzle;
};

// Encodes (or fetches from the cache) the tiled map described by `spec`.
// Returns false if the driver rejects it (bad alignment, stride or box).
bool get_tmap(const TmapSpec& spec, CUtensorMap* out);

}  // namespace mla
