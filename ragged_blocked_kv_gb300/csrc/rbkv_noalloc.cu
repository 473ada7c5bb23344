// Ragged attention for callers that cannot allocate device memory.
//
// Some callers of this library are not allowed to call cudaMalloc (or any
// allocator) at the point where they run attention: code that runs under a
// fixed memory budget handed out up front, code inside a runtime that owns
// all device memory through its own pool, or code running where an
// allocation could block or fail mid-step.  rbkv_ragged_attention needs a
// caller-provided workspace for the partial outputs of split decode rows;
// this entry point uses instead a scratch array that lives in the library
// itself, reserved when the library's device code is loaded.
//
// The scratch is a file-scope __device__ array of kStaticScratchBytes (16 MiB).
// Every GPU that loads the library holds it until the process exits.  All
// calls share the one array: calls whose kernels overlap on the GPU (for
// instance on two streams without ordering between them) race on it and give
// wrong results.  Nothing in it needs to start at zero: every partial slot a
// call reads is written earlier by the same call.
#include "rbkv.h"
#include "rbkv_internal.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];  // device address of the array, per device

}  // namespace

extern "C" rbkv_status rbkv_ragged_attention_noalloc(rbkv_pass* p, const void* q,
                                                     const void* k_cache, const void* v_cache,
                                                     void* o, rbkv_stream stream) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return rbkv::set_error(RBKV_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return rbkv::set_error(RBKV_ERR_UNSUPPORTED, "device index beyond the static scratch table");
  void* scratch = nullptr;
  {
    // One-time set-up per device, with that device current: the host-side
    // name of the array is not a device address, so ask the runtime for it.
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void* addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_static_scratch);
      if (e != cudaSuccess || !addr)
        return rbkv::set_error(RBKV_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
      g_scratch_addr[dev] = addr;
    }
    scratch = g_scratch_addr[dev];
  }
  return rbkv::attention_on_device(p, q, k_cache, v_cache, o, scratch, kStaticScratchBytes,
                                   (cudaStream_t)stream);
}
