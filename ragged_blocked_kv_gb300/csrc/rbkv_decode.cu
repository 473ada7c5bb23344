// Split-KV decode attention on the TMA + tensor-core path (filled in below).
#include "rbkv_internal.h"

namespace rbkv {

bool decode_fast_supported(const ShapeInfo&) { return false; }

cudaError_t launch_decode_fast(const DevPass&, const ShapeInfo&, const void*, const void*,
                               const void*, void*, float*, float*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace rbkv
