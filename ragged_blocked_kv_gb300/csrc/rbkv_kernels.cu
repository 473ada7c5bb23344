// kv_append, the CUDA-core attention path and the log-sum-exp combine.
//
// kv_append: FastGen guide, "Paged KV Memory Management" - new K/V rows go to
//   fixed-size blocks reached through the block table.  One warp per (token,
//   KV head) row pair: half the warp copies the K row, half the V row, with
//   coalesced 16-byte loads and stores.
// generic attention: exact softmax attention of one (row, KV head, key split)
//   work unit per CTA, online softmax over 32-key chunks (one key per lane),
//   fp32 arithmetic.  Used for fp32 layers and for shapes outside the
//   tensor-core kernels' envelope.
// combine: FastGen guide, "Two-Phase Softmax Reduction" and Step 3's split
//   path - partial outputs O_i with log-sum-exps L_i merge as
//   O = sum_i 2^(L_i - M) O_i / sum_i 2^(L_i - M), M = max_i L_i
//   (log-sum-exps are kept in base 2 inside the library).
#include <algorithm>

#include "rbkv_internal.h"
#include "rbkv_ptx.cuh"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace rbkv {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  atomicCAS(status, 0, code);
}

template <class T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <class T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// ---------------------------------------------------------------------------
// kv_append
// ---------------------------------------------------------------------------
// A flat copy of 16-byte vectors: vector i of the 2 * T * H_kv * (D / vec)
// new K and V vectors (K first, then V; inside each, the [T][H_kv][D] order of
// the input, so consecutive threads read consecutive addresses) goes to its
// token's cache slot.  Each thread keeps kAppendUnroll vectors in flight (all
// loads, data and slot ids, issued before the first store); the grid strides
// over the vectors, so one launch sized by a frame's capacity serves any pass.
constexpr int kAppendThreads = 256;
constexpr int kAppendUnroll = 4;

__global__ void __launch_bounds__(kAppendThreads)
    kv_append_kernel(DevPass dp, int32_t H_kv, int32_t B, int32_t vec_per_row,
                     const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     uint4* __restrict__ k_cache, uint4* __restrict__ v_cache) {
  // Launched to overlap its predecessor's tail: wait for it (it may have
  // produced k_new / v_new, or still read cache blocks this pass reuses).
  // The attention kernels may launch as soon as every CTA is here; they wait
  // for this grid before reading the cache.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t stride = gridDim.x * kAppendThreads;
  const uint32_t per_tok = (uint32_t)H_kv * (uint32_t)vec_per_row;
  const uint32_t half = (uint32_t)pass_count(dp, kCountTokens, dp.num_tokens) * per_tok;
  const uint32_t total = 2 * half;
  for (uint32_t i0 = blockIdx.x * kAppendThreads + threadIdx.x; i0 < total;
       i0 += kAppendUnroll * stride) {
    uint4 val[kAppendUnroll];
    int32_t slot[kAppendUnroll];
#pragma unroll
    for (int u = 0; u < kAppendUnroll; ++u) {
      const uint32_t i = i0 + u * stride;
      if (i < total) {
        const bool is_v = i >= half;
        const uint32_t j = is_v ? i - half : i;
        val[u] = is_v ? v_new[j] : k_new[j];
        slot[u] = dp.slot[j / per_tok];
      }
    }
#pragma unroll
    for (int u = 0; u < kAppendUnroll; ++u) {
      const uint32_t i = i0 + u * stride;
      if (i >= total) break;
      const bool is_v = i >= half;
      const uint32_t j = is_v ? i - half : i;
      const uint32_t hc = j % per_tok;
      const uint32_t h = hc / (uint32_t)vec_per_row, c = hc - h * (uint32_t)vec_per_row;
      const int32_t blk = slot[u] / B, off = slot[u] - blk * B;
      if (slot[u] < 0 || blk >= dp.num_blocks) {
        report(dp.status, kDevBounds);
        continue;
      }
      uint4* dst = is_v ? v_cache : k_cache;
      dst[(((size_t)blk * H_kv + h) * B + off) * vec_per_row + c] = val[u];
    }
  }
}

// ---------------------------------------------------------------------------
// metadata upload
// ---------------------------------------------------------------------------
// Copies a pass's packed metadata (status words, slots, block tables, work
// lists) from pinned host memory mapped into the device's address space to
// the pass's device buffer.  It is the first kernel of a pass, launched to
// overlap the previous pass's last kernel: each thread reads its vectors from
// host memory first, then waits for that kernel (the device buffer may be
// memory the previous passes used), then stores them.  A pass's upload is so
// part of the chain of kernels, with no copy between two passes' kernels.
constexpr int kUploadThreads = 256;
constexpr int kUploadUnroll = 4;

__global__ void __launch_bounds__(kUploadThreads)
    meta_upload_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int32_t vec) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t stride = gridDim.x * kUploadThreads;
  const uint32_t i0 = blockIdx.x * kUploadThreads + threadIdx.x;
  uint4 v[kUploadUnroll];
#pragma unroll
  for (int u = 0; u < kUploadUnroll; ++u) {
    const uint32_t i = i0 + u * stride;
    if (i < (uint32_t)vec) v[u] = src[i];
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll
  for (int u = 0; u < kUploadUnroll; ++u) {
    const uint32_t i = i0 + u * stride;
    if (i < (uint32_t)vec) dst[i] = v[u];
  }
}

// ---------------------------------------------------------------------------
// CUDA-core attention over one work unit per CTA
// ---------------------------------------------------------------------------
constexpr int kGenWarps = 4;
constexpr int kMaxDPerLane = 8;  // head_dim <= 256

template <class T>
__global__ void __launch_bounds__(kGenWarps * 32)
    generic_attention_kernel(DevPass dp, ShapeInfo s, const T* __restrict__ q,
                             const T* __restrict__ k_cache, const T* __restrict__ v_cache,
                             T* __restrict__ o, float* __restrict__ part_o,
                             float* __restrict__ part_lse) {
  __shared__ float q_s[kGenWarps][256];
  const WorkItem it = dp.generic_items[blockIdx.x];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int D = s.D, B = s.B, H_kv = s.H_kv;
  const int dpl = D / 32;  // elements of the output row per lane (D % 32 == 0 here)
  const float qscale = s.scale * kLog2e;
  const int32_t* table = dp.block_ids + it.table_off;

  for (int gi = warp; gi < s.g; gi += kGenWarps) {
    const int h = it.kv_head * s.g + gi;
    const T* qrow = q + ((int64_t)it.row * s.H_q + h) * D;
    for (int d = lane; d < D; d += 32) q_s[warp][d] = to_f(qrow[d]) * qscale;
    __syncwarp();

    float m = -INFINITY, l = 0.f;
    float acc[kMaxDPerLane];
#pragma unroll
    for (int i = 0; i < kMaxDPerLane; ++i) acc[i] = 0.f;

    for (int k0 = it.key_begin; k0 < it.key_end; k0 += 32) {
      const int key = k0 + lane;
      float sc = -INFINITY;
      int64_t row_off = -1;
      if (key < it.key_end) {
        const int32_t blk = table[key / B];
        if (blk >= 0 && blk < dp.num_blocks) {
          row_off = (((int64_t)blk * H_kv + it.kv_head) * B + key % B) * D;
          const T* krow = k_cache + row_off;
          float dot = 0.f;
          for (int d = 0; d < D; ++d) dot = fmaf(q_s[warp][d], to_f(krow[d]), dot);
          sc = dot;
        } else {
          report(dp.status, kDevBounds);
        }
      }
      float cmax = sc;
#pragma unroll
      for (int off = 16; off; off >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, off));
      const float m_new = fmaxf(m, cmax);
      if (m_new == -INFINITY) continue;  // every key of this chunk skipped
      const float corr = exp2f(m - m_new);
      const float p = exp2f(sc - m_new);
      float psum = p;
#pragma unroll
      for (int off = 16; off; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
      l = l * corr + psum;
#pragma unroll
      for (int i = 0; i < kMaxDPerLane; ++i) acc[i] *= corr;
      for (int j = 0; j < 32; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
        const int64_t roff = __shfl_sync(0xffffffffu, row_off, j);
        if (roff < 0) continue;
        const T* vrow = v_cache + roff;
#pragma unroll
        for (int i = 0; i < kMaxDPerLane; ++i)
          if (i < dpl) acc[i] = fmaf(pj, to_f(vrow[lane + 32 * i]), acc[i]);
      }
      m = m_new;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    if (it.part < 0) {
      T* orow = o + ((int64_t)it.row * s.H_q + h) * D;
#pragma unroll
      for (int i = 0; i < kMaxDPerLane; ++i)
        if (i < dpl) orow[lane + 32 * i] = from_f<T>(acc[i] * inv);
    } else {
      float* prow = part_o + ((int64_t)it.part * s.g + gi) * D;
#pragma unroll
      for (int i = 0; i < kMaxDPerLane; ++i)
        if (i < dpl) prow[lane + 32 * i] = acc[i] * inv;
      if (lane == 0) part_lse[(int64_t)it.part * s.g + gi] = l > 0.f ? m + log2f(l) : -INFINITY;
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// log-sum-exp combine: one warp per (split row, query head of the group)
// ---------------------------------------------------------------------------
// The lanes first read the row's log-sum-exps together (lane k takes splits
// k, k + 32, ...) for their maximum M and the weight sum; the weighted sum of
// the partial outputs then takes four splits per round, so that their loads
// are in flight together.
constexpr int kCombineSplitsInFlight = 4;

template <class T>
__global__ void __launch_bounds__(128)
    combine_kernel(DevPass dp, ShapeInfo s, const float* __restrict__ part_o,
                   const float* __restrict__ part_lse, T* __restrict__ o) {
  // launched to overlap the attention kernels' tail: the partials are only
  // complete once they have finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next pass's cache append may launch now (it waits for this grid)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x % 32;
  const int64_t n_warps = (int64_t)pass_count(dp, kCountCombine, dp.n_combine) * s.g;
  const int D = s.D, dpl = D / 32;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32; w < n_warps;
       w += (int64_t)gridDim.x * blockDim.x / 32) {
    const CombineRow cr = dp.combine_rows[w / s.g];
    const int gi = (int)(w % s.g);
    const float* lse = part_lse + (int64_t)cr.part_begin * s.g + gi;   // stride g per split
    float M = -INFINITY;
    for (int i = lane; i < cr.nsplit; i += 32) M = fmaxf(M, lse[(int64_t)i * s.g]);
#pragma unroll
    for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float wsum = 0.f;
    for (int i = lane; i < cr.nsplit; i += 32) {
      const float l = lse[(int64_t)i * s.g];
      wsum += (l == -INFINITY) ? 0.f : exp2f(l - M);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    float acc[kMaxDPerLane];
#pragma unroll
    for (int k = 0; k < kMaxDPerLane; ++k) acc[k] = 0.f;
    for (int i0 = 0; i0 < cr.nsplit; i0 += kCombineSplitsInFlight) {
      float wv[kCombineSplitsInFlight];
      float x[kCombineSplitsInFlight][kMaxDPerLane];
#pragma unroll
      for (int u = 0; u < kCombineSplitsInFlight; ++u) {
        const int i = i0 + u;
        wv[u] = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxDPerLane; ++k) x[u][k] = 0.f;
        if (i < cr.nsplit) {
          const float l = lse[(int64_t)i * s.g];
          wv[u] = (l == -INFINITY) ? 0.f : exp2f(l - M);
          const float* prow = part_o + ((int64_t)(cr.part_begin + i) * s.g + gi) * D;
#pragma unroll
          for (int k = 0; k < kMaxDPerLane; ++k)
            if (k < dpl) x[u][k] = prow[lane + 32 * k];
        }
      }
#pragma unroll
      for (int u = 0; u < kCombineSplitsInFlight; ++u)
#pragma unroll
        for (int k = 0; k < kMaxDPerLane; ++k) acc[k] = fmaf(wv[u], x[u][k], acc[k]);
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    T* orow = o + ((int64_t)cr.row * s.H_q + cr.kv_head * s.g + gi) * D;
#pragma unroll
    for (int k = 0; k < kMaxDPerLane; ++k)
      if (k < dpl) orow[lane + 32 * k] = from_f<T>(acc[k] * inv);
  }
}

int num_sms_current() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

}  // namespace

cudaError_t launch_kv_append(const DevPass& dp, const ShapeInfo& s, const void* k_new,
                             const void* v_new, void* k_cache, void* v_cache, cudaStream_t st,
                             bool overlap_previous) {
  const int esz = s.dtype == 0 ? 2 : 4;
  const int vec = s.D * esz / 16;
  const int64_t vectors = 2 * (int64_t)dp.num_tokens * s.H_kv * vec;
  if (vectors == 0) return cudaSuccess;
  if (vectors >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  // one wave: every thread takes kAppendUnroll vectors per round
  int64_t blocks = (vectors + kAppendThreads * kAppendUnroll - 1) / (kAppendThreads * kAppendUnroll);
  const int64_t cap = (int64_t)num_sms_current() * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kAppendThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kv_append_kernel, dp, s.H_kv, s.B, vec, (const uint4*)k_new,
                            (const uint4*)v_new, (uint4*)k_cache, (uint4*)v_cache);
}

cudaError_t launch_meta_upload(const void* src, void* dst, size_t bytes, cudaStream_t st,
                               bool overlap_previous) {
  if (bytes == 0) return cudaSuccess;
  if ((bytes & 15) || ((uintptr_t)src & 15) || ((uintptr_t)dst & 15))
    return cudaErrorMisalignedAddress;
  const int64_t vec = (int64_t)(bytes / 16);
  if (vec >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  // every thread holds kUploadUnroll vectors across the wait
  const int64_t blocks = (vec + kUploadThreads * kUploadUnroll - 1) / (kUploadThreads * kUploadUnroll);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kUploadThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, meta_upload_kernel, (const uint4*)src, (uint4*)dst,
                            (int32_t)vec);
}

cudaError_t launch_generic_attention(const DevPass& dp, const ShapeInfo& s, const void* q,
                                     const void* k_cache, const void* v_cache, void* o,
                                     float* part_o, float* part_lse, cudaStream_t st) {
  if (s.D % 32) return cudaErrorNotSupported;
  if (dp.n_generic == 0) return cudaSuccess;
  if (s.dtype == 0)
    generic_attention_kernel<__nv_bfloat16><<<dp.n_generic, kGenWarps * 32, 0, st>>>(
        dp, s, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k_cache,
        (const __nv_bfloat16*)v_cache, (__nv_bfloat16*)o, part_o, part_lse);
  else
    generic_attention_kernel<float><<<dp.n_generic, kGenWarps * 32, 0, st>>>(
        dp, s, (const float*)q, (const float*)k_cache, (const float*)v_cache, (float*)o, part_o,
        part_lse);
  return cudaGetLastError();
}

namespace {
__global__ void wait_timeout_kernel(int32_t* status, long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_barrier_init();
    if (!ptx::mbar_wait(&bar, 0, limit)) ptx::report_wait(status, kDevTimeout, 99, 0);
  }
}
}  // namespace

cudaError_t launch_wait_timeout(int32_t* status, long long limit, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status, limit);
  return cudaGetLastError();
}

cudaError_t launch_combine(const DevPass& dp, const ShapeInfo& s, const float* part_o,
                           const float* part_lse, void* o, cudaStream_t st) {
  if (s.D % 32) return cudaErrorNotSupported;
  const int64_t warps = (int64_t)dp.n_combine * s.g;
  if (warps == 0) return cudaSuccess;
  // one warp per (row, query head); a frame's capacity-sized launch strides
  int64_t nb = (warps * 32 + 127) / 128;
  if (dp.counts) nb = std::min<int64_t>(nb, (int64_t)num_sms_current() * 8);
  const unsigned blocks = (unsigned)nb;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (s.dtype == 0)
    return cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16>, dp, s, part_o, part_lse,
                              (__nv_bfloat16*)o);
  return cudaLaunchKernelEx(&cfg, combine_kernel<float>, dp, s, part_o, part_lse, (float*)o);
}

}  // namespace rbkv
