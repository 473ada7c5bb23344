// C ABI of the dense steps of a decoder layer: the tensor-core GEMM with its
// fused epilogues and RMSNorm (kernels in rbkv_gemm.cu).
#include "rbkv.h"
#include "rbkv_internal.h"

#include <string>

namespace {
rbkv_status invalid(const char* msg) { return rbkv::set_error(RBKV_ERR_INVALID, msg); }
bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }
}  // namespace

extern "C" {

size_t rbkv_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k) {
  if (m < 1 || n < 1 || k < 1) return 0;
  return rbkv::gemm_workspace_bytes(m, n, k);
}

rbkv_status rbkv_gemm_bf16(const void* a, const void* b, void* c, int64_t m, int64_t n, int64_t k,
                           const void* residual, int32_t epilogue, void* workspace,
                           size_t workspace_bytes, int32_t* status, rbkv_stream stream) {
  rbkv::NvtxRange nvtx_range("rbkv_gemm_bf16");
  if (m < 0 || n < 1 || k < 1) return invalid("m must be >= 0, n and k >= 1");
  if (m == 0) return RBKV_OK;
  if (!a || !b || !c) return invalid("NULL operand");
  if (m >= (1ll << 31) || n >= (1ll << 31) || k >= (1ll << 31))
    return invalid("sizes must fit in int32");
  if (k % 8) return invalid("k must be a multiple of 8 (16-byte rows)");
  if (!aligned16(a) || !aligned16(b) || !aligned16(c) || (residual && !aligned16(residual)))
    return invalid("operands must be 16-byte aligned");
  int64_t ldc = n;
  switch (epilogue) {
    case RBKV_GEMM_PLAIN:
      if (n % 32) return invalid("n must be a multiple of 32");
      break;
    case RBKV_GEMM_RESIDUAL:
      if (n % 32) return invalid("n must be a multiple of 32");
      if (!residual) return invalid("the residual epilogue needs a residual");
      break;
    case RBKV_GEMM_SWIGLU:
      if (n % 256) return invalid("the SwiGLU epilogue needs n a multiple of 256");
      ldc = n / 2;
      break;
    default:
      return invalid("unknown epilogue");
  }
  if (workspace && ((uintptr_t)workspace & 255)) return invalid("workspace must be 256-byte aligned");
  const size_t need = rbkv::gemm_workspace_bytes(m, n, k);
  const bool split = need > 0 && workspace && workspace_bytes >= need;
  cudaError_t e = rbkv::launch_gemm_bf16(a, b, c, residual, m, n, k, ldc, epilogue, status,
                                         (cudaStream_t)stream, nullptr, nullptr, 0, 0,
                                         split ? workspace : nullptr, split ? workspace_bytes : 0);
  if (e == cudaSuccess) rbkv::note_launches(split ? 2 : 1);
  if (e != cudaSuccess)
    return rbkv::set_error(RBKV_ERR_CUDA, (std::string("gemm launch: ") +
                                           cudaGetErrorString(e)).c_str());
  return RBKV_OK;
}

rbkv_status rbkv_gemm_bf16_qkv(const void* a, const void* w_qkv, void* q, void* k_out,
                               void* v_out, int64_t m, int64_t n_q, int64_t n_kv, int64_t k,
                               void* workspace, size_t workspace_bytes, int32_t* status,
                               rbkv_stream stream) {
  rbkv::NvtxRange nvtx_range("rbkv_gemm_bf16_qkv");
  if (m < 0 || n_q < 1 || n_kv < 1 || k < 1) return invalid("bad sizes");
  if (m == 0) return RBKV_OK;
  if (!a || !w_qkv || !q || !k_out || !v_out) return invalid("NULL operand");
  if (n_q % 32 || n_kv % 32) return invalid("n_q and n_kv must be multiples of 32");
  if (k % 8) return invalid("k must be a multiple of 8 (16-byte rows)");
  const int64_t n = n_q + 2 * n_kv;
  if (m >= (1ll << 31) || n >= (1ll << 31) || k >= (1ll << 31))
    return invalid("sizes must fit in int32");
  if (!aligned16(a) || !aligned16(w_qkv) || !aligned16(q) || !aligned16(k_out) || !aligned16(v_out))
    return invalid("operands must be 16-byte aligned");
  if (workspace && ((uintptr_t)workspace & 255)) return invalid("workspace must be 256-byte aligned");
  const size_t need = rbkv::gemm_workspace_bytes(m, n, k);
  const bool split = need > 0 && workspace && workspace_bytes >= need;
  cudaError_t e = rbkv::launch_gemm_bf16(a, w_qkv, q, nullptr, m, n, k, n_q, 3, status,
                                         (cudaStream_t)stream, k_out, v_out, n_q, n_q + n_kv,
                                         split ? workspace : nullptr, split ? workspace_bytes : 0);
  if (e == cudaSuccess) rbkv::note_launches(split ? 2 : 1);
  if (e != cudaSuccess)
    return rbkv::set_error(RBKV_ERR_CUDA, (std::string("gemm launch: ") +
                                           cudaGetErrorString(e)).c_str());
  return RBKV_OK;
}

rbkv_status rbkv_rmsnorm_bf16(const void* x, const void* weight, void* y, int64_t m,
                              int64_t hidden, float eps, rbkv_stream stream) {
  rbkv::NvtxRange nvtx_range("rbkv_rmsnorm_bf16");
  if (m < 0 || hidden < 8 || hidden % 8) return invalid("hidden must be a positive multiple of 8");
  if (m == 0) return RBKV_OK;
  if (!x || !weight || !y) return invalid("NULL tensor");
  if (!aligned16(x) || !aligned16(weight) || !aligned16(y)) return invalid("tensors must be 16-byte aligned");
  if (!(eps > 0.f)) return invalid("eps must be > 0");
  cudaError_t e = rbkv::launch_rmsnorm_bf16(x, weight, y, m, hidden, eps, (cudaStream_t)stream);
  if (e == cudaSuccess) rbkv::note_launches(1);
  if (e != cudaSuccess)
    return rbkv::set_error(RBKV_ERR_CUDA, (std::string("rmsnorm launch: ") +
                                           cudaGetErrorString(e)).c_str());
  return RBKV_OK;
}

}  // extern "C"
