// Prompt-chunk attention on tcgen05 tensor cores (filled in below).
#include "rbkv_internal.h"

namespace rbkv {

bool chunk_fast_supported(const ShapeInfo&) { return false; }

cudaError_t launch_chunk_fast(const DevPass&, const ShapeInfo&, const void*, const void*,
                              const void*, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace rbkv
