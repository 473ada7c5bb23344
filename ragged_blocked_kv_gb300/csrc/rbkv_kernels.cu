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
// One warp per (token, KV head): the first half of the warp copies the K row,
// the second half the V row, 16 bytes per lane per step (32-bit index math).
// A warp takes two rows at a time, with every load of both issued before the
// first store (rows are at most 64 x 16 bytes).
constexpr int kAppendWarps = 8;

__global__ void __launch_bounds__(kAppendWarps * 32)
    kv_append_kernel(DevPass dp, int32_t H_kv, int32_t B, int32_t vec_per_row,
                     const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     uint4* __restrict__ k_cache, uint4* __restrict__ v_cache) {
  // Launched to overlap its predecessor's tail: wait for it (it may have
  // produced k_new / v_new, or still read cache blocks this pass reuses).
  // The attention kernels may launch as soon as every CTA is here; they wait
  // for this grid before reading the cache.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, hl = lane & 15;
  const uint4* __restrict__ src = half ? v_new : k_new;
  uint4* __restrict__ dst = half ? v_cache : k_cache;
  const uint32_t rows = (uint32_t)pass_count(dp, kCountTokens, dp.num_tokens) * (uint32_t)H_kv;
  const uint32_t stride = gridDim.x * kAppendWarps;
  for (uint32_t r0 = blockIdx.x * kAppendWarps + warp; r0 < rows; r0 += 2 * stride) {
    const uint32_t r1 = r0 + stride;
    const bool two = r1 < rows;
    const uint32_t t0 = r0 / (uint32_t)H_kv;
    const uint32_t t1 = two ? r1 / (uint32_t)H_kv : t0;
    const int32_t slot0 = dp.slot[t0];
    const int32_t slot1 = dp.slot[t1];
    uint4 b0[4], b1[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int v = hl + 16 * i;
      if (v < vec_per_row) {
        b0[i] = src[(size_t)r0 * vec_per_row + v];
        if (two) b1[i] = src[(size_t)r1 * vec_per_row + v];
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (k == 1 && !two) break;
      const uint32_t r = k ? r1 : r0, t = k ? t1 : t0;
      const int32_t slot = k ? slot1 : slot0;
      const uint32_t h = r - t * (uint32_t)H_kv;
      const int32_t blk = slot / B, off = slot - blk * B;
      if (slot < 0 || blk >= dp.num_blocks) {
        if (lane == 0) report(dp.status, kDevBounds);
        continue;
      }
      uint4* d_row = dst + (((size_t)blk * H_kv + h) * B + off) * vec_per_row;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int v = hl + 16 * i;
        if (v < vec_per_row) d_row[v] = k ? b1[i] : b0[i];
      }
    }
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
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) / 32; w < n_warps;
       w += (int64_t)gridDim.x * blockDim.x / 32) {
  const CombineRow cr = dp.combine_rows[w / s.g];
  const int gi = (int)(w % s.g);
  const int D = s.D, dpl = D / 32;
  float M = -INFINITY;
  for (int i = 0; i < cr.nsplit; ++i) M = fmaxf(M, part_lse[(int64_t)(cr.part_begin + i) * s.g + gi]);
  float acc[kMaxDPerLane];
#pragma unroll
  for (int i = 0; i < kMaxDPerLane; ++i) acc[i] = 0.f;
  float wsum = 0.f;
  for (int i = 0; i < cr.nsplit; ++i) {
    const int64_t part = cr.part_begin + i;
    const float lse = part_lse[part * s.g + gi];
    const float wi = (lse == -INFINITY) ? 0.f : exp2f(lse - M);
    wsum += wi;
    const float* prow = part_o + (part * s.g + gi) * D;
#pragma unroll
    for (int k = 0; k < kMaxDPerLane; ++k)
      if (k < dpl) acc[k] = fmaf(wi, prow[lane + 32 * k], acc[k]);
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
  const int64_t rows = (int64_t)dp.num_tokens * s.H_kv;
  if (rows == 0) return cudaSuccess;
  if (rows >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  int64_t blocks = (rows + kAppendWarps - 1) / kAppendWarps;
  const int64_t cap = (int64_t)num_sms_current() * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kAppendWarps * 32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kv_append_kernel, dp, s.H_kv, s.B, vec, (const uint4*)k_new,
                            (const uint4*)v_new, (uint4*)k_cache, (uint4*)v_cache);
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
