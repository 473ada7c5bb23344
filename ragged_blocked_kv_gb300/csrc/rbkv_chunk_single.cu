// Prompt-chunk attention on the tensor cores, one query tile per CTA step
// (tcgen05).  The kernel for passes with few prompt-chunk tiles: every work
// item is one 128-row query tile of one query head (a work item of the
// paired kernel in rbkv_chunk.cu with no second tile).  With one tile, tensor
// memory has room for two score buffers, so the next key tile's QK^T runs
// while the softmax works on the current one; the paired kernel instead
// overlaps one tile's softmax with the other tile's products, which needs
// enough items to give every SM pairs.
//
// Roles (one CTA per SM, persistent over the items, which it walks in snake
// order, the planner having balanced the key-tile steps per CTA; barrier
// phases, the K/V ring and the score buffers carry over from item to item,
// tensor memory is allocated once):
//  - warp 4 (TMA): streams 128-key K and V tiles of the paged cache into a
//    3-stage ring (128-byte swizzle), looking block ids up a tile ahead;
//  - warp 5 (MMA): allocates 512 TMEM columns; one thread issues
//    S = Q K^T (M=128, N=128, K=128; Q in TMEM) into one of two TMEM S buffers
//    and O += P V (M=128, N=128, K=128; P in TMEM) into the TMEM O
//    accumulator, and signals completion with tcgen05.commit;
//  - warps 0-3 (softmax): thread i owns query row i = TMEM lane i; it writes
//    its row of Q into TMEM at the start of an item, reads its 128 scores with
//    tcgen05.ld (two halves), masks causally, keeps a running max that is
//    raised only when a row's max grows by more than 2^8 (the accumulator in
//    TMEM is then rescaled in place), writes P as bf16 pairs over the S
//    columns it has read, and finally normalises O and stores it.
// The QK^T of the next tile is queued on the tensor pipe before each PV, so it
// overlaps the softmax of the current one.  About 192 KB of shared memory.
// Every wait is bounded; on timeout the kernel records RBKV_ERR_TIMEOUT, lets
// its copies and MMAs drain (bounded), frees its TMEM and returns.
#include <algorithm>

#include <atomic>

#include "rbkv_internal.h"
#include "rbkv_ptx.cuh"
#include "rbkv_tcgen05.cuh"

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace rbkv {

namespace {

using namespace tc;

constexpr int kRows = kChunkTileRows;       // 128 query rows (MMA M)
constexpr int kKeys = kChunkTileKeys;       // 128 keys per KV tile (MMA N of QK^T)
constexpr int kStages = 3;
constexpr int kThreads = 6 * 32;
constexpr int kKVHalf = kKeys * 128;        // 16 KB: 128 keys x 64 head dims
constexpr int kKVTile = 2 * kKVHalf;        // 32 KB
constexpr int kStage = 2 * kKVTile;         // K + V
// Tensor memory (fp32 columns x 128 lanes, lane = query row): S0 [0,128) and
// S1 [128,256) (scores of one KV tile each), O [256,384), Q [384,448) as
// packed bf16 pairs (the QK^T A operand).  The probabilities P of a tile, as
// bf16 pairs (the PV A operand), overwrite the first 64 columns of its S
// buffer once they are read.
constexpr int kTmemCols = 512;
constexpr int kOCol = 256;
constexpr int kQCol = 384;
// 192 KB: one CTA per SM with a 3-deep ring of 128-key K/V tiles
constexpr int kSmemBytes = kStages * kStage + 256;
constexpr long long kWaitLimit = 4000000000LL;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

// Every barrier below is waited on in order of its phases and can never run
// two phases ahead of a waiter (the parity of a wait is then unambiguous): S,
// P and PV completion each have one barrier per buffer.
struct Bars {
  uint64_t q_full;      // the softmax threads wrote Q into tensor memory
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];   // QK^T of tile j done: S buffer j & 1
  uint64_t p_full[2];   // softmax of tile j done: P written over S buffer j & 1
  uint64_t o_done[2];   // PV of tile j done
  uint32_t tmem_base;
  int abort_flag;
};
// shared memory: K/V ring | barriers
static_assert(kStages * kStage + (int)sizeof(Bars) <= kSmemBytes,
              "shared-memory layout overflows its allocation");

__global__ void __launch_bounds__(kThreads, 1)
    chunk_single_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_k,
                              const __grid_constant__ CUtensorMap tmap_v, DevPass dp,
                              ShapeInfo shp, const __nv_bfloat16* __restrict__ q,
                              __nv_bfloat16* __restrict__ o,
                              float* __restrict__ part_o, float* __restrict__ part_lse,
                              int wait_first) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw;
  if (ptx::smem_u32(smem_raw) & 1023) {
    // the swizzled operand layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(dp.status, 0, kDevBounds);
    ptx::pdl_wait_previous();   // the grid's completion still covers its predecessor
    return;
  }
  uint8_t* kv_s = base;
  Bars* bars = reinterpret_cast<Bars*>(kv_s + kStages * kStage);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work items: one (tile, query head) each, sorted longest first; this
  // persistent CTA takes items in snake order over the grid
  const int n_items = pass_count(dp, kCountChunk, dp.n_chunk);
  if ((int)blockIdx.x >= n_items) {
    // a grid sized for a frame's capacity: nothing here.  Still wait for the
    // predecessor, so that this grid's completion covers it
    ptx::pdl_wait_previous();
    return;
  }
  const int G = gridDim.x;
  auto item_of = [&](int k) -> int {
    const int w = k * G + ((k & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
    return w < n_items ? w : -1;
  };
  const int B = shp.B;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->q_full, 4 * 32);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&bars->kv_full[s], 1);
      ptx::mbar_init(&bars->kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&bars->s_full[b], 1);
      ptx::mbar_init(&bars->p_full[b], 4 * 32);
      ptx::mbar_init(&bars->o_done[b], 1);
    }
    bars->abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // The grid may have been launched while its predecessor still runs.  After
  // the cache append (`wait_first`) it waits for it here, after the set-up.
  // After this call's decode kernel it need not: that kernel let it start
  // only once the append had finished; it then waits for the decode kernel
  // before ending, so that its completion covers both attention kernels.
  if (wait_first) ptx::pdl_wait_previous();
  if (threadIdx.x == 0) ptx::pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  // Every role walks the same items and KV tiles in the same order; `gi`
  // numbers this CTA's KV tiles across items, so the ring stage (gi % kStages),
  // the S/P buffer (gi & 1) and every barrier phase continue from item to item.
  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmap_k);
      ptx::tma_prefetch_desc(&tmap_v);
      const int box_rows = B < kKeys ? B : kKeys;
      uint32_t gi = 0;
      bool stop = false;
      for (int k = 0; !stop; ++k) {
        const int w = item_of(k);
        if (w < 0) break;
        const ChunkItem ci = dp.chunk_items[w];
        const ChunkTile tile = dp.chunk_tiles[ci.tile[0]];
        const int kvh = ci.kv_head;
        const int kb = tile.key_begin;
        const int ke = min(tile.key_end, tile.pos_begin + tile.n_rows);
        const int n_kv = (ke - kb + kKeys - 1) / kKeys;
        const int32_t* table = dp.block_ids + tile.table_off;
        // cache rows of the boxes of KV tile j (-1: out-of-range block,
        // skipped); looked up one tile ahead, so that the block-table loads
        // overlap the wait for a free stage
        int32_t rows[kKeys / 8];
        int nsub = 0, loads = 0;
        auto lookup = [&](int j) {
          nsub = 0;
          loads = 0;
          for (int r = 0; r < kKeys; r += box_rows) {
            const int key = kb + j * kKeys + r;
            if (key >= ke) break;
            const int32_t blk = table[key / B];
            if (blk < 0 || blk >= dp.num_blocks) {
              atomicCAS(dp.status, 0, kDevBounds);
              rows[nsub++] = -1;
              continue;
            }
            rows[nsub++] = (blk * shp.H_kv + kvh) * B + (key % B);
            ++loads;
          }
        };
        if (n_kv > 0) lookup(0);
        for (int j = 0; j < n_kv; ++j, ++gi) {
          const int s = gi % kStages;
          if (*abort_flag) {
            stop = true;
            break;
          }
          if (gi >= (uint32_t)kStages &&
              !ptx::mbar_wait(&bars->kv_empty[s], ((gi / kStages) - 1) & 1, kWaitLimit)) {
            ptx::report_wait(dp.status, kDevTimeout, 21, (int)gi);
            *abort_flag = 1;
            stop = true;
            break;
          }
          uint8_t* kdst = kv_s + s * kStage;
          uint8_t* vdst = kdst + kKVTile;
          ptx::mbar_arrive_expect_tx(&bars->kv_full[s], (uint32_t)(loads * box_rows * 128 * 4));
          for (int i = 0; i < nsub; ++i) {
            if (rows[i] < 0) continue;
            const int off = i * box_rows * 128;
            ptx::tma_load_2d(kdst + off, &tmap_k, 0, rows[i], &bars->kv_full[s]);
            ptx::tma_load_2d(kdst + kKVHalf + off, &tmap_k, 64, rows[i], &bars->kv_full[s]);
            ptx::tma_load_2d(vdst + off, &tmap_v, 0, rows[i], &bars->kv_full[s]);
            ptx::tma_load_2d(vdst + kKVHalf + off, &tmap_v, 64, rows[i], &bars->kv_full[s]);
          }
          if (j + 1 < n_kv) lookup(j + 1);
        }
      }
      // every copy must land before the CTA may exit
      for (uint32_t t = gi > (uint32_t)kStages ? gi - kStages : 0; t < gi; ++t)
        ptx::mbar_wait(&bars->kv_full[t % kStages], (t / kStages) & 1, kWaitLimit);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = instr_desc(kRows, kKeys, 0);
      constexpr uint32_t idesc_o = instr_desc(kRows, 128, 1);
      // descriptor words of ring stage 0 as K (K-major) and as V (MN-major,
      // halves kKVHalf apart); each MMA adds its offset to the low word
      const uint32_t hi = desc_hi(1024);
      const uint32_t k_lo = desc_lo(ptx::smem_u32(kv_s), 16);
      const uint32_t v_lo = desc_lo(ptx::smem_u32(kv_s) + kKVTile, kKVHalf);
      auto issue_qk = [&](uint32_t t) {
        const uint32_t kt = k_lo + (((t % kStages) * kStage) >> 4);
        const uint32_t d = tmem + (t & 1) * kKeys;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // head dims 16kk .. 16kk+15: Q columns 8kk.., K's half kk/4, 32-byte step kk%4;
          // N = all 128 keys of the tile
          const uint32_t ko = ((kk >> 2) * kKVHalf + (kk & 3) * 32) >> 4;
          tc_mma_ts_w(d, tmem + kQCol + kk * 8, kt + ko, hi, idesc_s, kk > 0);
        }
        tc_commit(&bars->s_full[t & 1]);
      };
      bool ok = true;
      int site = 0, at = 0;
      uint32_t gi = 0;
      long long pv_last = -1;   // the last PV issued (its tile number)
      for (int k = 0; ok; ++k) {
        const int w = item_of(k);
        if (w < 0) break;
        const ChunkTile tile = dp.chunk_tiles[dp.chunk_items[w].tile[0]];
        const int kb = tile.key_begin;
        const int ke = min(tile.key_end, tile.pos_begin + tile.n_rows);
        const int n_kv = (ke - kb + kKeys - 1) / kKeys;
        // this item's Q rows are in tensor memory
        if (!ptx::mbar_wait(&bars->q_full, k & 1, kWaitLimit) || *abort_flag) {
          ok = false;
          site = 22;
          at = k;
          break;
        }
        tc_fence_after();
        if (n_kv > 0) {
          if (!ptx::mbar_wait(&bars->kv_full[gi % kStages], (gi / kStages) & 1, kWaitLimit)) {
            ok = false;
            site = 23;
            at = (int)gi;
            break;
          }
          tc_fence_after();
          issue_qk(gi);
        }
        for (int j = 0; ok && j < n_kv; ++j) {
          const uint32_t t = gi + j;
          if (j + 1 < n_kv) {
            if (!ptx::mbar_wait(&bars->kv_full[(t + 1) % kStages], ((t + 1) / kStages) & 1,
                                kWaitLimit)) {
              ok = false;
              site = 24;
              at = (int)t + 1;
              break;
            }
            tc_fence_after();
            issue_qk(t + 1);
          }
          if (!ptx::mbar_wait(&bars->p_full[t & 1], (t >> 1) & 1, kWaitLimit) || *abort_flag) {
            ok = false;
            site = 25;
            at = (int)t;
            break;
          }
          tc_fence_after();
          const uint32_t vt = v_lo + (((t % kStages) * kStage) >> 4);
          const uint32_t pt = tmem + (t & 1) * kKeys;
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk) {
            // keys 16kk .. 16kk+15: P columns 8kk.., V rows 16kk.. (MN-major)
            tc_mma_ts_w(tmem + kOCol, pt + kk * 8, vt + ((kk * 2048) >> 4), hi, idesc_o,
                        j > 0 || kk > 0);
          }
          tc_commit(&bars->o_done[t & 1]);
          tc_commit(&bars->kv_empty[t % kStages]);
          pv_last = t;
        }
        gi += n_kv;
      }
      if (!ok) {
        ptx::report_wait(dp.status, kDevTimeout, site, at);
        *abort_flag = 1;
      }
      // the last PV (and so every earlier one) must finish before TMEM is released
      if (pv_last >= 0)
        ptx::mbar_wait(&bars->o_done[pv_last & 1], (pv_last >> 1) & 1, kWaitLimit);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int row = threadIdx.x;                      // 0..127 = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const float qk_scale = shp.scale * kLog2e;
    uint32_t gi = 0;
    bool ok = true;
    int site = 0, at = 0;
    for (int k = 0; ok; ++k) {
      const int w = item_of(k);
      if (w < 0) break;
      const ChunkItem ci = dp.chunk_items[w];
      const ChunkTile tile = dp.chunk_tiles[ci.tile[0]];
      const int h = ci.head[0];
      const int kvh = ci.kv_head;
      const int kb = tile.key_begin;
      const int ke = min(tile.key_end, tile.pos_begin + tile.n_rows);
      const int n_kv = (ke - kb + kKeys - 1) / kKeys;
      const int pos = tile.pos_begin + row;           // position of this query row
      {
        // this thread's query row -> tensor memory (the QK^T A operand); rows
        // past the tile's end are zero.  The previous item's MMAs have all
        // finished (its epilogue waited for its last PV).
        float qv[64];
        uint4* q4 = reinterpret_cast<uint4*>(qv);
        if (row < tile.n_rows) {
          const uint4* src = reinterpret_cast<const uint4*>(
              q + ((int64_t)(tile.row_begin + row) * shp.H_q + h) * 128);
#pragma unroll
          for (int i = 0; i < 16; ++i) q4[i] = src[i];
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) q4[i] = make_uint4(0, 0, 0, 0);
        }
        tmem_st32(lane_base + kQCol, qv);
        tmem_st32(lane_base + kQCol + 32, qv + 32);
        tmem_wait_st();
        tc_fence_before();
        ptx::mbar_arrive(&bars->q_full);
      }
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < n_kv; ++j) {
        const uint32_t t = gi + j;
        // tcgen05.ld/st are warp-collective: every decision below is warp-uniform
        const bool got = ptx::mbar_wait(&bars->s_full[t & 1], (t >> 1) & 1, kWaitLimit);
        if (!__all_sync(0xffffffffu, got) || __any_sync(0xffffffffu, *abort_flag != 0)) {
          ok = false;
          site = 31;
          at = (int)t;
          break;
        }
        tc_fence_after();
        const uint32_t s_col = lane_base + (t & 1) * kKeys;  // S of tile t; then its P
        const int key0 = kb + j * kKeys;
        // this row sees the tile's first `lim` keys: those <= its position and
        // before the split's end (a prefix of the tile, possibly empty or all)
        const int lim = min(pos + 1, ke) - key0;
        const bool full = __all_sync(0xffffffffu, lim >= kKeys);
        // row max over 8 independent partial maxima, in two 64-key halves (the
        // second half first, so that the first stays in registers)
        float sc[64];
        float mx8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx8[u] = -INFINITY;
#pragma unroll
        for (int hf = 1; hf >= 0; --hf) {
          tmem_ld32(s_col + hf * 64, sc);
          tmem_ld32(s_col + hf * 64 + 32, sc + 32);
          tmem_wait_ld();
          const int lh = lim - hf * 64;
          if (full) {
            // columns u, u+8, ..., u+56 into accumulator u: three-input maxima
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              float a = ptx::fmax3(mx8[u], sc[u], sc[u + 8]);
#pragma unroll
              for (int i = 0; i < 3; ++i) a = ptx::fmax3(a, sc[u + 16 + 16 * i], sc[u + 24 + 16 * i]);
              mx8[u] = a;
            }
          } else {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              mx8[c & 7] = fmaxf(mx8[c & 7], c < lh ? sc[c] : -INFINITY);
          }
        }
        const float mraw = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        // the scale is positive, so the row max scales with it
        const float mt = mraw * qk_scale;
        float corr = 1.f;
        const bool raise = mt > m_ref + kRescaleThreshold;
        if (raise) {
          corr = ptx::ex2(m_ref - mt);
          m_ref = mt;
        }
        // rescaling O needs every earlier PV of this item finished (only when
        // a row's max rose)
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
          const bool done =
              ptx::mbar_wait(&bars->o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, kWaitLimit);
          if (!__all_sync(0xffffffffu, done)) {
            ok = false;
            site = 33;
            at = (int)t;
            break;
          }
          tc_fence_after();
          {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              float ov[32];
              tmem_ld32(lane_base + kOCol + c4 * 32, ov);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c) ov[c] *= corr;
              tmem_st32(lane_base + kOCol + c4 * 32, ov);
            }
            tmem_wait_st();
          }
        }
        // a row with no key in this split so far keeps m_ref = -inf: its p are 0
        const float nbase = m_ref == -INFINITY ? 0.f : -m_ref;
        float ps8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) ps8[u] = 0.f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (hf == 1) {
            tmem_ld32(s_col + 64, sc);
            tmem_ld32(s_col + 96, sc + 32);
            tmem_wait_ld();
          }
          const int lh = lim - hf * 64;
          if (!full) {
#pragma unroll
            for (int c = 0; c < 64; ++c) sc[c] = c < lh ? sc[c] : -INFINITY;
          }
          // P of these 64 keys as bf16 pairs over S columns already read
          float pk[32];
          uint32_t* pk32 = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            // scaling and row sum as packed pairs: one instruction per two columns
            float x0, x1;
            ptx::fma2(x0, x1, sc[c], sc[c + 1], qk_scale, qk_scale, nbase, nbase);
            const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
            const int a = (c >> 1) & 3;
            ptx::add2(ps8[2 * a], ps8[2 * a + 1], p0, p1);
            pk32[c / 2] = ptx::pack_bf16x2(p0, p1);
          }
          tmem_st32(s_col + hf * 32, pk);
        }
        tmem_wait_st();
        const float ps =
            ((ps8[0] + ps8[1]) + (ps8[2] + ps8[3])) + ((ps8[4] + ps8[5]) + (ps8[6] + ps8[7]));
        l = l * corr + ps;
        if (j == n_kv - 1 && (ke % kKeys) != 0) {
          // keys past the split's end may be anything (unwritten slots): zero their V rows
          const int s = t % kStages;
          ptx::mbar_wait(&bars->kv_full[s], (t / kStages) & 1, kWaitLimit);
          uint8_t* vt = kv_s + s * kStage + kKVTile;
          const int valid = ke - key0;
          for (int e = row; e < (kKeys - valid) * 16; e += kRows) {
            const int key = valid + e / 16, c = e % 16;
            *reinterpret_cast<uint4*>(vt + (c >> 3) * kKVHalf + key * 128 + ((c & 7) << 4)) =
                make_uint4(0, 0, 0, 0);
          }
          // the PV MMA reads these rows through the async proxy
          ptx::fence_proxy_async_smem();
        }
        tc_fence_before();
        ptx::mbar_arrive(&bars->p_full[t & 1]);
      }
      bool fin = ok;
      if (fin && n_kv > 0) {
        const uint32_t tl = gi + n_kv - 1;
        fin = ptx::mbar_wait(&bars->o_done[tl & 1], (tl >> 1) & 1, kWaitLimit);
      }
      if (__all_sync(0xffffffffu, fin)) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const bool store = row < tile.n_rows;
        const bool partial = tile.part_base >= 0;
        __nv_bfloat16* orow = o + ((int64_t)(tile.row_begin + row) * shp.H_q + h) * 128;
        // partial slot of (row, KV head, split); query head h % g inside it
        const int64_t slot =
            ((int64_t)tile.part_base + ((int64_t)row * shp.H_kv + kvh) * tile.nsplit +
             tile.split) * shp.g + (h % shp.g);
        float* prow = part_o + slot * 128;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          float ov[32];
          if (n_kv > 0) {
            tmem_ld32(lane_base + kOCol + c4 * 32, ov);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = 0.f;   // an empty key range: no PV ran
          }
          if (store && !partial) {
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              uint4 v;
              v.x = ptx::pack_bf16x2(ov[c8 * 8 + 0] * inv, ov[c8 * 8 + 1] * inv);
              v.y = ptx::pack_bf16x2(ov[c8 * 8 + 2] * inv, ov[c8 * 8 + 3] * inv);
              v.z = ptx::pack_bf16x2(ov[c8 * 8 + 4] * inv, ov[c8 * 8 + 5] * inv);
              v.w = ptx::pack_bf16x2(ov[c8 * 8 + 6] * inv, ov[c8 * 8 + 7] * inv);
              *reinterpret_cast<uint4*>(orow + c4 * 32 + c8 * 8) = v;
            }
          } else if (store) {
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
              *reinterpret_cast<float4*>(prow + c4 * 32 + c8 * 4) =
                  make_float4(ov[c8 * 4 + 0] * inv, ov[c8 * 4 + 1] * inv, ov[c8 * 4 + 2] * inv,
                              ov[c8 * 4 + 3] * inv);
          }
        }
        if (store && partial) part_lse[slot] = l > 0.f ? m_ref + log2f(l) : -INFINITY;
      } else {
        if (ok) {
          ok = false;
          site = 34;
          at = (int)(gi + n_kv);
        }
      }
      gi += n_kv;
    }
    if (!ok) {
      ptx::report_wait(dp.status, kDevTimeout, site, at);
      *abort_flag = 1;
    }
  }

  // all roles done (every wait above is bounded): release TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (!wait_first) ptx::pdl_wait_previous();
}

}  // namespace

cudaError_t launch_chunk_single(const DevPass& dp, const ShapeInfo& s, const void* q,
                              const void* k_cache, const void* v_cache, void* o, float* part_o,
                              float* part_lse, cudaStream_t st, bool overlap_previous,
                              bool wait_first) {
  if (dp.n_chunk == 0) return cudaSuccess;
  if (((uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache) & 15)
    return cudaErrorMisalignedAddress;
  const int64_t rows = (int64_t)dp.num_blocks * s.H_kv * s.B;
  const int box_rows = s.B < kKeys ? s.B : kKeys;
  CUtensorMap tk, tv;
  cudaError_t e = make_cache_tmap(&tk, k_cache, rows, s.D, box_rows);
  if (e == cudaSuccess) e = make_cache_tmap(&tv, v_cache, rows, s.D, box_rows);
  if (e != cudaSuccess) return e;
  // the shared-memory limit is raised once per device
  static std::atomic<uint64_t> attr_done{0};
  int attr_dev = 0;
  e = cudaGetDevice(&attr_dev);
  if (e != cudaSuccess) return e;
  const uint64_t attr_bit = 1ull << (attr_dev & 63);
  if (!(attr_done.load() & attr_bit)) {
    e = cudaFuncSetAttribute(chunk_single_tcgen05_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(chunk_single_tcgen05_kernel,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(attr_bit);
  }
  // persistent: at most one CTA per SM, each walking (tile, head) items
  static int sms_of[64] = {0};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int sms = dev < 64 ? sms_of[dev] : 0;
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) sms_of[dev] = sms;
  }
  dim3 grid((unsigned)std::min<int64_t>(dp.n_chunk, std::max(1, sms)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_previous ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, chunk_single_tcgen05_kernel, tk, tv, dp, s,
                            (const __nv_bfloat16*)q, (__nv_bfloat16*)o, part_o, part_lse,
                            wait_first ? 1 : 0);
}

}  // namespace rbkv
