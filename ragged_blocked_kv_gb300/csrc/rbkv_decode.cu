// Split-KV decode attention: one query token per (sequence, KV head, key
// split), all query heads of the KV head's group at once (FastGen guide,
// "Dynamic SplitKV Attention": each split computes a partial output and its
// log-sum-exp; Step 3's split path shows the per-split softmax).
//
// GB300 design (HBM-bound: every cached K/V byte is read once):
//  - persistent grid, one CTA per SM, each CTA walks a host-ordered list of
//    work units (longest first, dealt in snake order so CTAs finish together);
//  - a producer warp streams 64-key K and V tiles of the paged cache with TMA
//    (2-D tiled loads through the block table, 128-byte swizzle) into a
//    5-stage shared-memory ring guarded by mbarriers;
//  - four consumer warps take the tiles of a unit in turn; each multiplies the
//    group's query rows (padded to 16) by the tile with warp-level bf16 MMAs
//    (fp32 accumulation), runs the online softmax in registers with quad
//    shuffles, and accumulates P.V with MMAs;
//  - at the end of a unit the four warps merge their (max, sum, O) states in
//    shared memory and write either O (bf16) or the fp32 partial output and
//    base-2 log-sum-exp for the combine kernel.
// Every wait is bounded: on timeout the kernel records RBKV_ERR_TIMEOUT in the
// pass's status word and stops.
#include "rbkv_internal.h"
#include "rbkv_ptx.cuh"

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

namespace rbkv {

namespace {

constexpr int kStages = 5;
constexpr int kConsumers = 4;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kKeys = kDecodeTileKeys;        // 64 keys per tile
constexpr int kHalf = kKeys * 128;            // 64 rows x 128 B (64 bf16 of head_dim)
constexpr int kTile = 2 * kHalf;              // K or V tile, head_dim 128
constexpr int kStage = 2 * kTile;             // K + V
constexpr int kRowPad = 132;                  // fp32 row stride of the merge scratch
constexpr int kScratchBytes = kConsumers * 16 * kRowPad * 4;
constexpr int kMlBytes = kConsumers * 16 * 2 * 4;
constexpr int kSmemBytes = 1024 /*align slack*/ + kStages * kStage + kScratchBytes + kMlBytes +
                           2 * kStages * 8;
constexpr long long kWaitLimit = 4000000000LL;   // ~2 s of SM clock
constexpr float kLog2e = 1.4426950408889634f;

struct Shared {
  uint8_t* stages;     // kStages x kStage, 1024-aligned
  float* scratch;      // [kConsumers][16][kRowPad]
  float* ml;           // [kConsumers][16][2]
  uint64_t* full;      // [kStages]
  uint64_t* empty;     // [kStages]
};

__device__ __forceinline__ Shared carve(uint8_t* raw) {
  Shared s;
  uintptr_t base = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023);
  s.stages = reinterpret_cast<uint8_t*>(base);
  s.scratch = reinterpret_cast<float*>(s.stages + kStages * kStage);
  s.ml = s.scratch + kConsumers * 16 * kRowPad;
  s.full = reinterpret_cast<uint64_t*>(s.ml + kConsumers * 16 * 2);
  s.empty = s.full + kStages;
  return s;
}

__device__ __forceinline__ int tiles_of(const WorkItem& it) {
  return (it.key_end - it.key_begin + kKeys - 1) / kKeys;
}

// Byte offset, inside one K or V tile, of the 16-byte chunk holding elements
// d..d+7 (d % 8 == 0) of key row `key` (TMA 128-byte swizzle: chunk index XOR
// row index mod 8, each 64-column half a separate 8 KB box).
__device__ __forceinline__ uint32_t tile_off(int key, int d) {
  const int half = d >> 6;
  const int chunk = (d & 63) >> 3;
  return half * kHalf + key * 128 + ((chunk ^ (key & 7)) << 4);
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_splitkv_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, DevPass dp, ShapeInfo shp,
                          const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ o,
                          float* __restrict__ part_o, float* __restrict__ part_lse) {
  extern __shared__ uint8_t smem_raw[];
  Shared sm = carve(smem_raw);
  volatile __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = shp.g, B = shp.B, H_kv = shp.H_kv;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&sm.full[s], 1);
      ptx::mbar_init(&sm.empty[s], 1);
    }
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmap_k);
      ptx::tma_prefetch_desc(&tmap_v);
      uint32_t idx = 0;
      const int box_rows = B < kKeys ? B : kKeys;
      for (int item = blockIdx.x; item < dp.n_decode && !abort_flag; item += gridDim.x) {
        const WorkItem it = dp.decode_items[item];
        const int32_t* table = dp.block_ids + it.table_off;
        const int nt = tiles_of(it);
        for (int j = 0; j < nt; ++j, ++idx) {
          const int s = idx % kStages;
          if (idx >= (uint32_t)kStages &&
              !ptx::mbar_wait(&sm.empty[s], ((idx / kStages) - 1) & 1, kWaitLimit)) {
            atomicCAS(dp.status, 0, kDevTimeout);
            abort_flag = 1;
            break;
          }
          const int k0 = it.key_begin + j * kKeys;
          uint8_t* kdst = sm.stages + s * kStage;
          uint8_t* vdst = kdst + kTile;
          // sub-boxes of box_rows keys; skip those past the unit's last key
          int nsub = 0;
          int32_t rows[kKeys / 8];
          for (int r = 0; r < kKeys; r += box_rows) {
            const int key = k0 + r;
            if (key >= it.key_end) break;
            const int32_t blk = table[key / B];
            if (blk < 0 || blk >= dp.num_blocks) {
              atomicCAS(dp.status, 0, kDevBounds);
              rows[nsub++] = -1;
              continue;
            }
            rows[nsub++] = (blk * H_kv + it.kv_head) * B + (key % B);
          }
          int loads = 0;
          for (int i = 0; i < nsub; ++i) loads += rows[i] >= 0;
          ptx::mbar_arrive_expect_tx(&sm.full[s], (uint32_t)(loads * box_rows * 128 * 4));
          for (int i = 0; i < nsub; ++i) {
            if (rows[i] < 0) continue;
            const int off = i * box_rows * 128;
            ptx::tma_load_2d(kdst + off, &tmap_k, 0, rows[i], &sm.full[s]);
            ptx::tma_load_2d(kdst + kHalf + off, &tmap_k, 64, rows[i], &sm.full[s]);
            ptx::tma_load_2d(vdst + off, &tmap_v, 0, rows[i], &sm.full[s]);
            ptx::tma_load_2d(vdst + kHalf + off, &tmap_v, 64, rows[i], &sm.full[s]);
          }
        }
        if (abort_flag) break;
      }
      // let every load this CTA issued land before the CTA can exit
      const uint32_t issued = idx;
      for (uint32_t t = issued > (uint32_t)kStages ? issued - kStages : 0; t < issued; ++t)
        ptx::mbar_wait(&sm.full[t % kStages], (t / kStages) & 1, kWaitLimit);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const float qk_scale = shp.scale * kLog2e;
  const int r0 = lane >> 2, r1 = r0 + 8;      // fragment rows (query heads of the group)
  const int cq = (lane & 3) * 2;              // fragment column pair
  uint32_t tile_base = 0;
  const uint32_t stages_u32 = ptx::smem_u32(sm.stages);

  for (int item = blockIdx.x; item < dp.n_decode; item += gridDim.x) {
    const WorkItem it = dp.decode_items[item];
    const int nt = tiles_of(it);

    // query rows of the group as m16n8k16 A fragments (rows >= g are zero)
    uint32_t qa[8][4];
    {
      const __nv_bfloat16* qbase = q + ((int64_t)it.row * shp.H_q + it.kv_head * g) * 128;
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(qbase + r0 * 128);
      const uint32_t* q1 = reinterpret_cast<const uint32_t*>(qbase + r1 * 128);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int c = (kk * 16 + cq) >> 1;
        qa[kk][0] = r0 < g ? __ldg(q0 + c) : 0u;
        qa[kk][1] = r1 < g ? __ldg(q1 + c) : 0u;
        qa[kk][2] = r0 < g ? __ldg(q0 + c + 4) : 0u;
        qa[kk][3] = r1 < g ? __ldg(q1 + c + 4) : 0u;
      }
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc_o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc_o[i][0] = acc_o[i][1] = acc_o[i][2] = acc_o[i][3] = 0.f;

    for (int j = warp; j < nt && !abort_flag; j += kConsumers) {
      const uint32_t idx = tile_base + j;
      const int s = idx % kStages;
      if (!ptx::mbar_wait(&sm.full[s], (idx / kStages) & 1, kWaitLimit)) {
        // give up on this unit; the merge barriers below are still met by
        // every consumer warp, then all of them leave together
        if (lane == 0) { atomicCAS(dp.status, 0, kDevTimeout); abort_flag = 1; }
        __syncwarp();
        break;
      }
      const int k0 = it.key_begin + j * kKeys;
      const int valid = min(kKeys, it.key_end - k0);
      const uint32_t kt = stages_u32 + s * kStage;
      const uint32_t vt = kt + kTile;
      if (valid < kKeys) {
        // rows past the unit's last key may hold anything (unwritten cache
        // slots, stale tiles): zero their V rows so 0 * V stays 0
        uint8_t* vrow = sm.stages + s * kStage + kTile;
        for (int e = lane; e < (kKeys - valid) * 16; e += 32) {
          const int key = valid + e / 16, c = e % 16;
          *reinterpret_cast<uint4*>(vrow + (c >> 3) * kHalf + key * 128 + ((c & 7) << 4)) =
              make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }

      // S = Q K^T over the 64 keys: 8 n-tiles of 8 keys
      float sc[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int mi = lane >> 3;
          const int key = np * 16 + (mi >> 1) * 8 + (lane & 7);
          const int d = kk * 16 + (mi & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ptx::ldsm_x4(kt + tile_off(key, d), b0, b1, b2, b3);
          ptx::mma_bf16_16816(sc[2 * np], qa[kk], b0, b1);
          ptx::mma_bf16_16816(sc[2 * np + 1], qa[kk], b2, b3);
        }
      }
      // scale, mask keys past the unit, online softmax (rows r0 and r1)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int key = n * 8 + cq;
        sc[n][0] = key < valid ? sc[n][0] * qk_scale : -INFINITY;
        sc[n][1] = key + 1 < valid ? sc[n][1] * qk_scale : -INFINITY;
        sc[n][2] = key < valid ? sc[n][2] * qk_scale : -INFINITY;
        sc[n][3] = key + 1 < valid ? sc[n][3] * qk_scale : -INFINITY;
        mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float c0 = exp2f(m0 - mn0), c1 = exp2f(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.f, ps1 = 0.f;
      uint32_t pa[4][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const float p0 = exp2f(sc[n][0] - mn0), p1 = exp2f(sc[n][1] - mn0);
        const float p2 = exp2f(sc[n][2] - mn1), p3 = exp2f(sc[n][3] - mn1);
        ps0 += p0 + p1;
        ps1 += p2 + p3;
        pa[n >> 1][(n & 1) * 2 + 0] = ptx::pack_bf16x2(p0, p1);
        pa[n >> 1][(n & 1) * 2 + 1] = ptx::pack_bf16x2(p2, p3);
      }
      l0 = l0 * c0 + ps0;
      l1 = l1 * c1 + ps1;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        acc_o[i][0] *= c0;
        acc_o[i][1] *= c0;
        acc_o[i][2] *= c1;
        acc_o[i][3] *= c1;
      }
      // O += P V: 4 k-steps of 16 keys, 16 n-tiles of 8 head-dim columns
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int dp2 = 0; dp2 < 8; ++dp2) {
          const int mi = lane >> 3;
          const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
          const int d = dp2 * 16 + (mi >> 1) * 8;
          uint32_t b0, b1, b2, b3;
          ptx::ldsm_x4_t(vt + tile_off(key, d), b0, b1, b2, b3);
          ptx::mma_bf16_16816(acc_o[2 * dp2], pa[kk], b0, b1);
          ptx::mma_bf16_16816(acc_o[2 * dp2 + 1], pa[kk], b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) {
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(&sm.empty[s]);
      }
    }
    tile_base += nt;

    // ---- merge the four warps' states and write the unit's result -------
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if ((lane & 3) == 0) {
      sm.ml[(warp * 16 + r0) * 2 + 0] = m0;
      sm.ml[(warp * 16 + r0) * 2 + 1] = l0;
      sm.ml[(warp * 16 + r1) * 2 + 0] = m1;
      sm.ml[(warp * 16 + r1) * 2 + 1] = l1;
    }
    ptx::named_bar_sync(1, kConsumers * 32);
    float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) {
      M0 = fmaxf(M0, sm.ml[(w * 16 + r0) * 2]);
      M1 = fmaxf(M1, sm.ml[(w * 16 + r1) * 2]);
    }
    float L0 = 0.f, L1 = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) {
      const float mw0 = sm.ml[(w * 16 + r0) * 2], mw1 = sm.ml[(w * 16 + r1) * 2];
      if (mw0 != -INFINITY) L0 += exp2f(mw0 - M0) * sm.ml[(w * 16 + r0) * 2 + 1];
      if (mw1 != -INFINITY) L1 += exp2f(mw1 - M1) * sm.ml[(w * 16 + r1) * 2 + 1];
    }
    const float f0 = (m0 == -INFINITY || L0 == 0.f) ? 0.f : exp2f(m0 - M0) / L0;
    const float f1 = (m1 == -INFINITY || L1 == 0.f) ? 0.f : exp2f(m1 - M1) / L1;
    float* scr = sm.scratch + warp * 16 * kRowPad;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int d = i * 8 + cq;
      if (r0 < g)
        *reinterpret_cast<float2*>(scr + r0 * kRowPad + d) =
            make_float2(acc_o[i][0] * f0, acc_o[i][1] * f0);
      if (r1 < g)
        *reinterpret_cast<float2*>(scr + r1 * kRowPad + d) =
            make_float2(acc_o[i][2] * f1, acc_o[i][3] * f1);
    }
    ptx::named_bar_sync(1, kConsumers * 32);
    const int t = threadIdx.x;   // 0..127
    for (int e = t; e < g * 32; e += kConsumers * 32) {
      const int r = e >> 5, c4 = (e & 31) * 4;
      float4 a = *reinterpret_cast<const float4*>(sm.scratch + r * kRowPad + c4);
#pragma unroll
      for (int w = 1; w < kConsumers; ++w) {
        const float4 b = *reinterpret_cast<const float4*>(sm.scratch + (w * 16 + r) * kRowPad + c4);
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      if (it.part < 0) {
        __nv_bfloat16* orow = o + ((int64_t)it.row * shp.H_q + it.kv_head * g + r) * 128 + c4;
        uint2 packed;
        packed.x = ptx::pack_bf16x2(a.x, a.y);
        packed.y = ptx::pack_bf16x2(a.z, a.w);
        *reinterpret_cast<uint2*>(orow) = packed;
      } else {
        *reinterpret_cast<float4*>(part_o + ((int64_t)it.part * g + r) * 128 + c4) = a;
      }
    }
    if (it.part >= 0 && t < g) {
      float M = -INFINITY, L = 0.f;
      for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, sm.ml[(w * 16 + t) * 2]);
      for (int w = 0; w < kConsumers; ++w) {
        const float mw = sm.ml[(w * 16 + t) * 2];
        if (mw != -INFINITY) L += exp2f(mw - M) * sm.ml[(w * 16 + t) * 2 + 1];
      }
      part_lse[(int64_t)it.part * g + t] = L > 0.f ? M + log2f(L) : -INFINITY;
    }
    ptx::named_bar_sync(1, kConsumers * 32);
    if (abort_flag) return;
  }
}

// ---- host: tensor maps -------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

// Rows of a [num_blocks][H_kv][B][head_dim] bf16 cache as a 2-D tensor
// (head_dim columns), boxes of 64 columns x box_rows rows, 128-byte swizzle.
cudaError_t make_cache_tmap(CUtensorMap* m, const void* cache, int64_t rows, int head_dim,
                            int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool decode_fast_supported(const ShapeInfo& s) {
  const bool block_ok = (s.B % kKeys == 0) || (kKeys % s.B == 0 && s.B % 8 == 0);
  return s.dtype == 0 && s.D == 128 && s.g >= 1 && s.g <= 16 && block_ok;
}

cudaError_t launch_decode_fast(const DevPass& dp, const ShapeInfo& s, const void* q,
                               const void* k_cache, const void* v_cache, void* o, float* part_o,
                               float* part_lse, cudaStream_t st) {
  if (!decode_fast_supported(s)) return cudaErrorNotSupported;
  if (dp.n_decode == 0) return cudaSuccess;
  if (((uintptr_t)k_cache | (uintptr_t)v_cache) & 15) return cudaErrorMisalignedAddress;
  const int64_t rows = (int64_t)dp.num_blocks * s.H_kv * s.B;
  const int box_rows = s.B < kKeys ? s.B : kKeys;
  CUtensorMap tk, tv;
  cudaError_t e = make_cache_tmap(&tk, k_cache, rows, s.D, box_rows);
  if (e == cudaSuccess) e = make_cache_tmap(&tv, v_cache, rows, s.D, box_rows);
  if (e != cudaSuccess) return e;
  static bool attr_done = false;
  if (!attr_done) {
    e = cudaFuncSetAttribute(decode_splitkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  decode_splitkv_kernel<<<dp.decode_grid, kThreads, kSmemBytes, st>>>(
      tk, tv, dp, s, (const __nv_bfloat16*)q, (__nv_bfloat16*)o, part_o, part_lse);
  return cudaGetLastError();
}

}  // namespace rbkv
