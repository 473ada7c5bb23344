// Split-KV decode attention: one query token per (sequence, KV head, key
// split), all query heads of the KV head's group at once (FastGen guide,
// "Dynamic SplitKV Attention": each split computes a partial output and its
// log-sum-exp; Step 3's split path shows the per-split softmax).
//
// GB300 design (HBM-bound: every cached K/V byte is read once):
//  - persistent grid, two CTAs per SM (one for groups above 8 query heads),
//    each CTA walks a host-ordered list of work units (longest first, dealt in
//    snake order so CTAs finish together);
//  - a producer warp streams 64-key K and V tiles of the paged cache with TMA
//    (2-D tiled loads through the block table, 128-byte swizzle) into a
//    3-stage shared-memory ring guarded by mbarriers (six tiles in flight per
//    SM, and two CTAs' consumers to hide each other's latency);
//  - four consumer warps share every tile, 16 keys each (so each warp consumes
//    the ring strictly in order); each multiplies the group's query rows
//    (padded to 16) by its keys with warp-level bf16 MMAs (fp32 accumulation),
//    runs the online softmax in registers with quad shuffles, and accumulates
//    P.V with MMAs;
//  - at the end of a unit the four warps merge their (max, sum, O) states in
//    shared memory and write either O (bf16) or the fp32 partial output and
//    base-2 log-sum-exp for the combine kernel.
// Every wait is bounded: on timeout the kernel records RBKV_ERR_TIMEOUT in the
// pass's status word and stops.
#include <atomic>

#include "rbkv_internal.h"
#include "rbkv_ptx.cuh"

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

namespace rbkv {

namespace {

constexpr int kStages = 3;
constexpr int kConsumers = 4;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kKeys = kDecodeTileKeys;        // 64 keys per tile
constexpr int kHalf = kKeys * 128;            // 64 rows x 128 B (64 bf16 of head_dim)
constexpr int kTile = 2 * kHalf;              // K or V tile, head_dim 128
constexpr int kStage = 2 * kTile;             // K + V
constexpr int kRowPad = 132;                  // fp32 row stride of the merge scratch
// Rows of a unit's merge buffers: its query rows x heads - g for decode rows;
// with packed prompt rows (`packed`), up to kDecodeRowsCap for groups of up
// to kDecodeRowsCap heads, g above that.
__host__ __device__ constexpr int rows_cap_for(int g, bool packed) {
  return packed && g < kDecodeRowsCap ? kDecodeRowsCap : g;
}
// a 3-deep ring of 32 KB K+V tiles, the merge scratch [warp][rows][kRowPad]
// fp32, (max, sum) per warp and row, barriers: 96.6 KB (g = 1) to 112.8 KB
// (g = 8, or packed rows) - two CTAs per SM - and 129.2 KB for g = 16 (one)
__host__ __device__ constexpr int smem_bytes_for(int g, bool packed) {
  return kStages * kStage + kConsumers * rows_cap_for(g, packed) * (kRowPad + 2) * 4 +
         2 * kStages * 8 + 16;
}
constexpr int kMaxSmemBytes = smem_bytes_for(16, true);
constexpr long long kWaitLimit = 4000000000LL;   // ~2 s of SM clock
constexpr float kLog2e = 1.4426950408889634f;

struct Shared {
  uint8_t* stages;     // kStages x kStage, 1024-aligned
  float* scratch;      // [kConsumers][rows][kRowPad]
  float* ml;           // [kConsumers][rows][2]
  uint64_t* full;      // [kStages]
  uint64_t* empty;     // [kStages]
  volatile int* abort_flag;
};

// shared memory: K/V ring | merge buffer | (max, sum) per warp and row |
// full and empty barriers | abort flag (smem_bytes_for(g) bytes)
__device__ __forceinline__ Shared carve(uint8_t* raw, int rows) {
  Shared s;
  s.stages = raw;
  s.scratch = reinterpret_cast<float*>(s.stages + kStages * kStage);
  s.ml = s.scratch + kConsumers * rows * kRowPad;
  s.full = reinterpret_cast<uint64_t*>(s.ml + kConsumers * rows * 2);
  s.empty = s.full + kStages;
  s.abort_flag = reinterpret_cast<volatile int*>(s.empty + kStages);
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

template <bool kPacked>
__global__ void __launch_bounds__(kThreads, 2)
    decode_splitkv_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, DevPass dp, ShapeInfo shp,
                          const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ o,
                          float* __restrict__ part_o, float* __restrict__ part_lse,
                          int wait_first) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The kernel runs first among a pass's attention kernels.  With
  // `wait_first` it waits for its predecessor (the cache append) before any
  // global access, and only then lets the next kernel (prompt chunks, or the
  // combine) launch: that kernel may then read the cache without a wait of
  // its own.  It waits for its predecessor again before ending (needed when
  // it was launched without `wait_first`), so that its completion covers it.
  if (wait_first) ptx::pdl_wait_previous();
  ptx::pdl_launch_dependents();
  const int rcap = rows_cap_for(shp.g, kPacked);
  Shared sm = carve(smem_raw, rcap);
  volatile int& abort_flag = *sm.abort_flag;
  const int n_decode = pass_count(dp, kCountDecode, dp.n_decode);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = shp.g, B = shp.B, H_kv = shp.H_kv;
  if (ptx::smem_u32(smem_raw) & 1023) {
    // the swizzled tile layout needs a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(dp.status, 0, kDevBounds);
    ptx::pdl_wait_previous();   // the grid's completion still covers its predecessor
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&sm.full[s], 1);
      ptx::mbar_init(&sm.empty[s], kConsumers);
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
      for (int item = blockIdx.x; item < n_decode && !abort_flag; item += gridDim.x) {
        const WorkItem it = dp.decode_items[item];
        const int32_t* table = dp.block_ids + it.table_off;
        const int nt = tiles_of(it);
        for (int j = 0; j < nt; ++j, ++idx) {
          const int s = idx % kStages;
          if (idx >= (uint32_t)kStages &&
              !ptx::mbar_wait(&sm.empty[s], ((idx / kStages) - 1) & 1, kWaitLimit)) {
            ptx::report_wait(dp.status, kDevTimeout, 11, (int)idx);
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
    ptx::pdl_wait_previous();
    return;
  }

  // -------------------------------------------------------------- consumers
  const float qk_scale = shp.scale * kLog2e;
  const int r0 = lane >> 2, r1 = r0 + 8;      // fragment rows (query heads of the group)
  const int cq = (lane & 3) * 2;              // fragment column pair
  uint32_t tile_base = 0;
  const uint32_t stages_u32 = ptx::smem_u32(sm.stages);

  // the query rows of a unit as m16n8k16 A fragments: fragment row r is
  // query head r % g of the unit's row r / g; rows past n_rows * g are zero
  auto load_q = [&](int item, uint32_t(&dst)[8][4]) {
    const WorkItem u = dp.decode_items[item];
    const int nrg = kPacked ? u.n_rows * g : g;
    const __nv_bfloat16* qb0 =
        q + ((int64_t)(u.row + r0 / g) * shp.H_q + u.kv_head * g + r0 % g) * 128;
    const __nv_bfloat16* qb1 =
        q + ((int64_t)(u.row + r1 / g) * shp.H_q + u.kv_head * g + r1 % g) * 128;
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(qb0);
    const uint32_t* q1 = reinterpret_cast<const uint32_t*>(qb1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int c = (kk * 16 + cq) >> 1;
      dst[kk][0] = r0 < nrg ? __ldg(q0 + c) : 0u;
      dst[kk][1] = r1 < nrg ? __ldg(q1 + c) : 0u;
      dst[kk][2] = r0 < nrg ? __ldg(q0 + c + 4) : 0u;
      dst[kk][3] = r1 < nrg ? __ldg(q1 + c + 4) : 0u;
    }
  };
  uint32_t qa[8][4];
  if ((int)blockIdx.x < n_decode) load_q(blockIdx.x, qa);

  for (int item = blockIdx.x; item < n_decode; item += gridDim.x) {
    const WorkItem it = dp.decode_items[item];
    const int nt = tiles_of(it);
    const int nrg = kPacked ? it.n_rows * g : g;
    // keys visible to fragment rows r0 and r1 (packed rows are causal)
    const int lim0 = kPacked && r0 < nrg ? min(it.key_end, it.diag + r0 / g) : it.key_end;
    const int lim1 = kPacked && r1 < nrg ? min(it.key_end, it.diag + r1 / g) : it.key_end;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float acc_o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc_o[i][0] = acc_o[i][1] = acc_o[i][2] = acc_o[i][3] = 0.f;

    // every warp takes 16 keys (rows 16*warp .. 16*warp+15) of every tile, so
    // each warp consumes the stages strictly in order
    const int wk = warp * 16;
    for (int j = 0; j < nt && !abort_flag; ++j) {
      const uint32_t idx = tile_base + j;
      const int s = idx % kStages;
      if (!ptx::mbar_wait(&sm.full[s], (idx / kStages) & 1, kWaitLimit)) {
        // give up on this unit; the merge barriers below are still met by
        // every consumer warp, then all of them leave together
        if (lane == 0) {
          ptx::report_wait(dp.status, kDevTimeout, 12, (int)idx);
          abort_flag = 1;
        }
        __syncwarp();
        break;
      }
      const int k0 = it.key_begin + j * kKeys;
      const int valid = min(kKeys, it.key_end - k0) - wk;   // valid keys of this warp's 16
      const uint32_t kt = stages_u32 + s * kStage;
      const uint32_t vt = kt + kTile;
      if (valid < 16) {
        // rows past the unit's last key may hold anything (unwritten cache
        // slots, stale tiles): zero this warp's such V rows so 0 * V stays 0
        uint8_t* vrow = sm.stages + s * kStage + kTile;
        const int first = valid < 0 ? 0 : valid;
        for (int e = lane; e < (16 - first) * 16; e += 32) {
          const int key = wk + first + e / 16, c = e % 16;
          *reinterpret_cast<uint4*>(vrow + (c >> 3) * kHalf + key * 128 + ((c & 7) << 4)) =
              make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      if (valid > 0) {
        // S = Q K^T over this warp's 16 keys: 2 n-tiles of 8 keys
        float sc[2][4];
        sc[0][0] = sc[0][1] = sc[0][2] = sc[0][3] = 0.f;
        sc[1][0] = sc[1][1] = sc[1][2] = sc[1][3] = 0.f;
        const int mi = lane >> 3;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int key = wk + (mi >> 1) * 8 + (lane & 7);
          const int d = kk * 16 + (mi & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ptx::ldsm_x4(kt + tile_off(key, d), b0, b1, b2, b3);
          ptx::mma_bf16_16816(sc[0], qa[kk], b0, b1);
          ptx::mma_bf16_16816(sc[1], qa[kk], b2, b3);
        }
        // scale, mask keys past each row's limit, online softmax (rows r0 and r1)
        const int valid0 = min(kKeys, lim0 - k0) - wk, valid1 = min(kKeys, lim1 - k0) - wk;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          const int key = n * 8 + cq;
          sc[n][0] = key < valid0 ? sc[n][0] * qk_scale : -INFINITY;
          sc[n][1] = key + 1 < valid0 ? sc[n][1] * qk_scale : -INFINITY;
          sc[n][2] = key < valid1 ? sc[n][2] * qk_scale : -INFINITY;
          sc[n][3] = key + 1 < valid1 ? sc[n][3] * qk_scale : -INFINITY;
          mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
          mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        // a row with no visible key so far keeps max -inf: its terms are 0
        const float b0 = mn0 == -INFINITY ? 0.f : mn0, b1 = mn1 == -INFINITY ? 0.f : mn1;
        const float c0 = ptx::ex2(m0 - b0), c1 = ptx::ex2(m1 - b1);
        m0 = mn0;
        m1 = mn1;
        const float p00 = ptx::ex2(sc[0][0] - b0), p01 = ptx::ex2(sc[0][1] - b0);
        const float p02 = ptx::ex2(sc[0][2] - b1), p03 = ptx::ex2(sc[0][3] - b1);
        const float p10 = ptx::ex2(sc[1][0] - b0), p11 = ptx::ex2(sc[1][1] - b0);
        const float p12 = ptx::ex2(sc[1][2] - b1), p13 = ptx::ex2(sc[1][3] - b1);
        l0 = l0 * c0 + (p00 + p01 + p10 + p11);
        l1 = l1 * c1 + (p02 + p03 + p12 + p13);
        uint32_t pa[4];
        pa[0] = ptx::pack_bf16x2(p00, p01);
        pa[1] = ptx::pack_bf16x2(p02, p03);
        pa[2] = ptx::pack_bf16x2(p10, p11);
        pa[3] = ptx::pack_bf16x2(p12, p13);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          acc_o[i][0] *= c0;
          acc_o[i][1] *= c0;
          acc_o[i][2] *= c1;
          acc_o[i][3] *= c1;
        }
        // O += P V over the 16 keys: 16 n-tiles of 8 head-dim columns
#pragma unroll
        for (int dp2 = 0; dp2 < 8; ++dp2) {
          const int key = wk + (mi & 1) * 8 + (lane & 7);
          const int d = dp2 * 16 + (mi >> 1) * 8;
          uint32_t b0, b1, b2, b3;
          ptx::ldsm_x4_t(vt + tile_off(key, d), b0, b1, b2, b3);
          ptx::mma_bf16_16816(acc_o[2 * dp2], pa, b0, b1);
          ptx::mma_bf16_16816(acc_o[2 * dp2 + 1], pa, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) {
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(&sm.empty[s]);
      }
    }
    tile_base += nt;

    // the next unit's queries, loaded while this one is merged
    uint32_t qn[8][4];
    const int next = item + gridDim.x;
    if (next < n_decode) load_q(next, qn);

    // ---- merge the four warps' states and write the unit's result -------
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    // (fragment rows >= n_rows * g are padding: they take no part)
    if ((lane & 3) == 0) {
      if (r0 < nrg) {
        sm.ml[(warp * rcap + r0) * 2 + 0] = m0;
        sm.ml[(warp * rcap + r0) * 2 + 1] = l0;
      }
      if (r1 < nrg) {
        sm.ml[(warp * rcap + r1) * 2 + 0] = m1;
        sm.ml[(warp * rcap + r1) * 2 + 1] = l1;
      }
    }
    ptx::named_bar_sync(1, kConsumers * 32);
    float M0 = -INFINITY, M1 = -INFINITY;
    float L0 = 0.f, L1 = 0.f;
    if (r0 < nrg) {
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) M0 = fmaxf(M0, sm.ml[(w * rcap + r0) * 2]);
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        const float mw0 = sm.ml[(w * rcap + r0) * 2];
        if (mw0 != -INFINITY) L0 += ptx::ex2(mw0 - M0) * sm.ml[(w * rcap + r0) * 2 + 1];
      }
    }
    if (r1 < nrg) {
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) M1 = fmaxf(M1, sm.ml[(w * rcap + r1) * 2]);
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        const float mw1 = sm.ml[(w * rcap + r1) * 2];
        if (mw1 != -INFINITY) L1 += ptx::ex2(mw1 - M1) * sm.ml[(w * rcap + r1) * 2 + 1];
      }
    }
    const float f0 = (m0 == -INFINITY || L0 == 0.f) ? 0.f : ptx::ex2(m0 - M0) / L0;
    const float f1 = (m1 == -INFINITY || L1 == 0.f) ? 0.f : ptx::ex2(m1 - M1) / L1;
    // each warp stores its rescaled O; then all four are summed per element
    float* scr = sm.scratch + warp * rcap * kRowPad;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int d = i * 8 + cq;
      if (r0 < nrg)
        *reinterpret_cast<float2*>(scr + r0 * kRowPad + d) =
            make_float2(acc_o[i][0] * f0, acc_o[i][1] * f0);
      if (r1 < nrg)
        *reinterpret_cast<float2*>(scr + r1 * kRowPad + d) =
            make_float2(acc_o[i][2] * f1, acc_o[i][3] * f1);
    }
    ptx::named_bar_sync(1, kConsumers * 32);
    const int t = threadIdx.x;   // 0..127
    for (int e = t; e < nrg * 32; e += kConsumers * 32) {
      const int r = e >> 5, c4 = (e & 31) * 4;
      float4 a = *reinterpret_cast<const float4*>(sm.scratch + r * kRowPad + c4);
#pragma unroll
      for (int w = 1; w < kConsumers; ++w) {
        const float4 b =
            *reinterpret_cast<const float4*>(sm.scratch + (w * rcap + r) * kRowPad + c4);
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      if (it.part < 0) {
        __nv_bfloat16* orow =
            o + ((int64_t)(it.row + r / g) * shp.H_q + it.kv_head * g + r % g) * 128 + c4;
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
      for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, sm.ml[(w * rcap + t) * 2]);
      for (int w = 0; w < kConsumers; ++w) {
        const float mw = sm.ml[(w * rcap + t) * 2];
        if (mw != -INFINITY) L += ptx::ex2(mw - M) * sm.ml[(w * rcap + t) * 2 + 1];
      }
      part_lse[(int64_t)it.part * g + t] = L > 0.f ? M + log2f(L) : -INFINITY;
    }
    // all consumer warps leave together if anyone gave up
    if (ptx::named_bar_or(1, kConsumers * 32, abort_flag != 0)) break;
    if (next < n_decode) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
#pragma unroll
        for (int x = 0; x < 4; ++x) qa[kk][x] = qn[kk][x];
    }
  }
  ptx::pdl_wait_previous();
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

// A row-major bf16 matrix [rows][cols] as a 2-D TMA tensor: boxes of 64
// columns (128 bytes) x box_rows rows, 128-byte swizzle; rows past the end
// read as zero.  A descriptor depends only on these arguments, and a serving
// loop passes the same cache arrays for every pass, so the last few encoded
// descriptors are kept per host thread and reused.
cudaError_t make_tmap_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols,
                         int box_rows) {
  struct Entry {
    CUtensorMap map;
    const void* ptr;
    int64_t rows, cols;
    int box_rows;
  };
  constexpr int kEntries = 8;
  thread_local Entry cache[kEntries];
  thread_local int filled = 0, next = 0;
  for (int i = 0; i < filled; ++i) {
    const Entry& e = cache[i];
    if (e.ptr == ptr && e.rows == rows && e.cols == cols && e.box_rows == box_rows) {
      *m = e.map;
      return cudaSuccess;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  Entry& e = cache[next];
  e.map = *m;
  e.ptr = ptr;
  e.rows = rows;
  e.cols = cols;
  e.box_rows = box_rows;
  next = (next + 1) % kEntries;
  if (filled < kEntries) ++filled;
  return cudaSuccess;
}

cudaError_t make_cache_tmap(CUtensorMap* m, const void* cache, int64_t rows, int head_dim,
                            int box_rows) {
  return make_tmap_2d(m, cache, rows, head_dim, box_rows);
}

int decode_ctas_per_sm(const ShapeInfo& s) {
  // two CTAs fit when each leaves room for the other (228 KB per SM, 1 KB
  // reserved per CTA; 160 threads x at most 204 registers each)
  return 2 * (smem_bytes_for(s.g, true) + 1024) <= 228 * 1024 ? 2 : 1;
}

bool decode_fast_supported(const ShapeInfo& s) {
  const bool block_ok = (s.B % kKeys == 0) || (kKeys % s.B == 0 && s.B % 8 == 0);
  return s.dtype == 0 && s.D == 128 && s.g >= 1 && s.g <= 16 && block_ok;
}

cudaError_t launch_decode_fast(const DevPass& dp, const ShapeInfo& s, const void* q,
                               const void* k_cache, const void* v_cache, void* o, float* part_o,
                               float* part_lse, cudaStream_t st, bool overlap_previous,
                               bool wait_first) {
  if (!decode_fast_supported(s)) return cudaErrorNotSupported;
  if (dp.n_decode == 0) return cudaSuccess;
  if (((uintptr_t)k_cache | (uintptr_t)v_cache) & 15) return cudaErrorMisalignedAddress;
  const int64_t rows = (int64_t)dp.num_blocks * s.H_kv * s.B;
  const int box_rows = s.B < kKeys ? s.B : kKeys;
  CUtensorMap tk, tv;
  cudaError_t e = make_cache_tmap(&tk, k_cache, rows, s.D, box_rows);
  if (e == cudaSuccess) e = make_cache_tmap(&tv, v_cache, rows, s.D, box_rows);
  if (e != cudaSuccess) return e;
  // the shared-memory limit of each variant is raised once per device
  static std::atomic<uint64_t> attr_done{0};
  int attr_dev = 0;
  e = cudaGetDevice(&attr_dev);
  if (e != cudaSuccess) return e;
  const uint64_t attr_bit = 1ull << (attr_dev & 63);
  if (!(attr_done.load() & attr_bit)) {
    for (int v = 0; v < 2 && e == cudaSuccess; ++v) {
      auto fn = v ? decode_splitkv_kernel<true> : decode_splitkv_kernel<false>;
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemBytes);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    }
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(attr_bit);
  }
  const bool packed = dp.decode_packed != 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(dp.decode_grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes_for(s.g, packed);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  return cudaLaunchKernelEx(&cfg,
                            packed ? decode_splitkv_kernel<true> : decode_splitkv_kernel<false>,
                            tk, tv, dp, s, (const __nv_bfloat16*)q, (__nv_bfloat16*)o, part_o,
                            part_lse, wait_first ? 1 : 0);
}

}  // namespace rbkv
