// Prompt-chunk attention on the fifth-generation tensor cores (tcgen05).
//
// FastGen guide, "The Continuous Batching Dilemma": prompt processing is a
// dense contraction that belongs on the tensor cores.  A chunk row at position
// p attends keys 0..p of its sequence: the cached prefix read through the
// block table plus the chunk's own earlier rows (causal within the chunk).
//
// A work item is one or two 128-row query tiles that read the same K/V tiles:
// the same rows for two query heads of one KV group (K/V then cross HBM once
// for both), or two consecutive row tiles of one head when a group has one
// head.  A persistent grid of one CTA per SM walks the items in snake order,
// which the planner fills so that every CTA gets about the same number of
// key-tile steps; barrier phases, the K/V ring and tensor memory carry over
// from item to item.  Roles:
//  - warp 8 (TMA): loads each item's query tiles (A and B) into shared memory
//    and streams 128-key K and V tiles of the paged cache, in the order
//    K0 V0 K1 V1 ..., through a 5-stage ring of 32 KB stages (128-byte
//    swizzle), looking block ids up through the block table;
//  - warp 9 (MMA): one thread issues, per query tile X, S_X = Q_X K^T
//    (M=128, N=128 keys, K=128; Q from shared memory) into tensor memory and
//    O_X += P_X V (M=128, N=128 head dims, K=128 keys; P from tensor memory),
//    in the order QK_A(0) QK_B(0), then for each key tile j: PV_A(j)
//    QK_A(j+1) PV_B(j) QK_B(j+1).  Each tile's products follow its softmax,
//    so one tile's softmax runs while the tensor pipe works on the other
//    tile (an issuing thread per tile was measured slower: interleaved, each
//    tile's products take longer to finish);
//  - warps 0-3 / 4-7 (softmax of tile A / B): thread i owns query row i = TMEM
//    lane i: it reads its 128 scores with tcgen05.ld (one round trip), masks
//    causally, keeps a running max that is raised only when the row max grows
//    by more than 2^8 (the accumulator in tensor memory is then rescaled in
//    place), writes P as bf16 pairs over the score columns it has read, and at
//    the end of an item normalises O and stores it (or the partial output and
//    its log-sum-exp when the item covers one piece of a split key range).
// Tensor memory (512 columns x 128 lanes): S/P of A [0,128), O of A
// [128,256), S/P of B [256,384), O of B [384,512).  Shared memory: Q of A and
// B (32 KB each) and the ring (160 KB), about 225 KB: one CTA per SM.  Each
// group of eight MMAs (K = 128) is issued from one instruction block.
// Every wait is bounded; on timeout the kernel records RBKV_ERR_TIMEOUT, lets
// its copies and MMAs drain (bounded), frees its tensor memory and returns.
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
constexpr int kStages = 5;                  // ring stages, each one K or one V tile
constexpr int kHalf = kKeys * 128;          // 16 KB: 128 rows x 64 head dims
constexpr int kTileBytes = 2 * kHalf;       // 32 KB: 128 rows x 128 head dims
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
// three warpgroups: two softmax warpgroups and one with the TMA and MMA
// warps (its other two warps idle), so that registers can move between
// warpgroups:
// launched at kLaunchRegs a thread, the third warpgroup gives back down to
// kIssueRegs and the softmax warpgroups take kSoftmaxRegs.  The shares add up
// to the launch's total exactly (a larger claim would wait forever).
constexpr int kThreads = 12 * 32;
constexpr int kLaunchRegs = 168;
constexpr int kIssueRegs = 88;
constexpr int kSoftmaxRegs = 208;
static_assert(128 * kIssueRegs + 256 * kSoftmaxRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch's registers");
constexpr int kTmemCols = 512;
constexpr int kTileCols = 256;              // tensor-memory columns of one query tile
constexpr int kOCol = 128;                  // O after S/P inside a tile's columns
constexpr int kSmemBytes = 2 * kTileBytes + kStages * kTileBytes + 1024;
constexpr long long kWaitLimit = 4000000000LL;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

// Each barrier is waited on in order of its phases and can never run two
// phases ahead of a waiter (the parity of a wait is then unambiguous).
struct Bars {
  uint64_t q_full[2];    // query tile X landed (TMA)
  uint64_t q_empty[2];   // the last QK^T of an item read query tile X
  uint64_t kv_full[kStages];      // a K or V tile landed (TMA)
  uint64_t kv_empty[kStages];     // the MMAs are done with the stage
  uint64_t s_full[2];    // QK^T of tile X done: S_X readable
  uint64_t p_full[2];    // softmax of tile X done: P_X written (and V tail rows zeroed)
  uint64_t o_done[2];    // PV of tile X done
  uint64_t drain;        // every MMA the CTA issued done (before tensor memory is freed)
  uint64_t o_free[2];    // epilogue of tile X read O_X: the next item may overwrite it
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(2 * kTileBytes + kStages * kTileBytes + (int)sizeof(Bars) <= kSmemBytes,
              "shared-memory layout overflows its allocation");

// An item as every role sees it (each role reads the rest of a query tile's
// description itself, when it needs it).
struct Item {
  int tile[2];     // chunk tile of each query tile (-1: none)
  int head[2];
  int n[2];        // key tiles of each query tile (0: no such tile)
  int kv_head;
  int kb, ke;      // key range of the item (the union of its tiles')
  int nmax;        // key tiles of the item
};

__device__ __forceinline__ Item load_item(const DevPass& dp, int w) {
  const ChunkItem ci = dp.chunk_items[w];
  Item it;
  it.kv_head = ci.kv_head;
  it.kb = ci.key_begin;
  it.ke = ci.key_end;
  it.nmax = (it.ke - it.kb + kKeys - 1) / kKeys;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    it.tile[x] = ci.tile[x];
    it.head[x] = ci.head[x];
    it.n[x] = ci.tile[x] >= 0
                  ? (dp.chunk_tiles[ci.tile[x]].key_end - it.kb + kKeys - 1) / kKeys
                  : 0;
  }
  return it;
}

__global__ void __launch_bounds__(kThreads, 1)
    chunk_attn_tcgen05_kernel(const __grid_constant__ CUtensorMap tmap_q,
                              const __grid_constant__ CUtensorMap tmap_k,
                              const __grid_constant__ CUtensorMap tmap_v, DevPass dp,
                              ShapeInfo shp, __nv_bfloat16* __restrict__ o,
                              float* __restrict__ part_o, float* __restrict__ part_lse,
                              int wait_first) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (ptx::smem_u32(smem_raw) & 1023) {
    // the swizzled operand layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(dp.status, 0, kDevBounds);
    ptx::pdl_wait_previous();   // the grid's completion still covers its predecessor
    return;
  }
  uint8_t* q_s = smem_raw;                       // [2][kTileBytes]
  uint8_t* kv_s = smem_raw + 2 * kTileBytes;     // [kStages][kTileBytes]
  Bars* bars = reinterpret_cast<Bars*>(kv_s + kStages * kTileBytes);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(&bars->q_full[x], 1);
      ptx::mbar_init(&bars->q_empty[x], 1);
      ptx::mbar_init(&bars->s_full[x], 1);
      ptx::mbar_init(&bars->p_full[x], 4 * 32);
      ptx::mbar_init(&bars->o_done[x], 1);
      if (x == 0) ptx::mbar_init(&bars->drain, 1);
      ptx::mbar_init(&bars->o_free[x], 4 * 32);
    }
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&bars->kv_full[s], 1);
      ptx::mbar_init(&bars->kv_empty[s], 1);
    }
    bars->abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == kMmaWarp) {
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

  // Every role walks the same items in the same order.  The ring index `gi`
  // numbers this CTA's K and V tiles across items (K_j of an item at 2j, V_j
  // at 2j + 1 from the item's start), so stages and phases carry over.
  if (warp >= 8) {
  // the TMA, MMA and V warps' warpgroup gives registers to the softmax warpgroups
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kIssueRegs));
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmap_q);
      ptx::tma_prefetch_desc(&tmap_k);
      ptx::tma_prefetch_desc(&tmap_v);
      const int box_rows = B < kKeys ? B : kKeys;
      uint32_t gi = 0, qi[2] = {0, 0};
      bool stop = false;
      for (int k = 0; !stop; ++k) {
        const int w = item_of(k);
        if (w < 0) break;
        const Item it = load_item(dp, w);
        #pragma unroll
        for (int x = 0; x < 2 && !stop; ++x) {
          if (it.n[x] == 0) continue;
          if (qi[x] > 0 &&
              !ptx::mbar_wait(&bars->q_empty[x], (qi[x] - 1) & 1, kWaitLimit)) {
            ptx::report_wait(dp.status, kDevTimeout, 41, k);
            *abort_flag = 1;
            stop = true;
            break;
          }
          uint8_t* dst = q_s + x * kTileBytes;
          const int row0 = dp.chunk_tiles[it.tile[x]].row_begin;
          ptx::mbar_arrive_expect_tx(&bars->q_full[x], kTileBytes);
          ptx::tma_load_2d(dst, &tmap_q, it.head[x] * 128, row0, &bars->q_full[x]);
          ptx::tma_load_2d(dst + kHalf, &tmap_q, it.head[x] * 128 + 64, row0, &bars->q_full[x]);
          ++qi[x];
        }
        const int32_t* table = dp.block_ids + dp.chunk_tiles[it.tile[0]].table_off;
        for (int j = 0; j < it.nmax && !stop; ++j) {
          // the boxes of key tile j: box i holds keys key0 + i * box_rows ..; a
          // box whose block id is out of range is skipped (and reported).  Rows
          // are recomputed where needed rather than kept in an array (a
          // runtime-indexed array would live in local memory)
          const int key0 = it.kb + j * kKeys;
          const int nsub = (min(it.ke - key0, kKeys) + box_rows - 1) / box_rows;
          auto box_row = [&](int i) -> int {
            const int key = key0 + i * box_rows;
            const int32_t blk = table[key / B];
            if (blk < 0 || blk >= dp.num_blocks) return -1;
            return (blk * shp.H_kv + it.kv_head) * B + (key % B);
          };
          int loads = 0;
          for (int i = 0; i < nsub; ++i) {
            if (box_row(i) >= 0)
              ++loads;
            else
              atomicCAS(dp.status, 0, kDevBounds);
          }
          for (int kv = 0; kv < 2; ++kv, ++gi) {
            const int s = gi % kStages;
            if (*abort_flag) {
              stop = true;
              break;
            }
            if (gi >= (uint32_t)kStages &&
                !ptx::mbar_wait(&bars->kv_empty[s], ((gi / kStages) - 1) & 1, kWaitLimit)) {
              ptx::report_wait(dp.status, kDevTimeout, 42, (int)gi);
              *abort_flag = 1;
              stop = true;
              break;
            }
            const CUtensorMap* map = kv ? &tmap_v : &tmap_k;
            uint8_t* dst = kv_s + s * kTileBytes;
            ptx::mbar_arrive_expect_tx(&bars->kv_full[s], (uint32_t)(loads * box_rows * 128 * 2));
            for (int i = 0; i < nsub; ++i) {
              const int row = box_row(i);
              if (row < 0) continue;
              const int off = i * box_rows * 128;
              ptx::tma_load_2d(dst + off, map, 0, row, &bars->kv_full[s]);
              ptx::tma_load_2d(dst + kHalf + off, map, 64, row, &bars->kv_full[s]);
            }
          }
        }
      }
      // every copy must land before the CTA may exit
      for (uint32_t t = gi > (uint32_t)kStages ? gi - kStages : 0; t < gi; ++t)
        ptx::mbar_wait(&bars->kv_full[t % kStages], (t / kStages) & 1, kWaitLimit);
      #pragma unroll
      for (int x = 0; x < 2; ++x)
        if (qi[x] > 0) ptx::mbar_wait(&bars->q_full[x], (qi[x] - 1) & 1, kWaitLimit);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = instr_desc(kRows, kKeys, 0);
      constexpr uint32_t idesc_o = instr_desc(kRows, 128, 1);
      // descriptor words: the high word is common to every operand; the low
      // words of the Q tiles and of ring stage 0 (as K, K-major, and as V,
      // MN-major with the two 64-column halves kHalf apart) are offset per MMA
      const uint32_t hi = desc_hi(1024);
      const uint32_t q_lo = desc_lo(ptx::smem_u32(q_s), 16);
      const uint32_t k_lo = desc_lo(ptx::smem_u32(kv_s), 16);
      const uint32_t v_lo = desc_lo(ptx::smem_u32(kv_s), kHalf);
      // S_X = Q_X K^T into tile X's S columns (after the previous PV of tile X
      // read P_X over the same columns: MMAs of one thread run in order)
      auto issue_qk = [&](int x, uint32_t gk, bool last) {
        const uint32_t qt = q_lo + ((x * kTileBytes) >> 4);
        const uint32_t kt = k_lo + (((gk % kStages) * kTileBytes) >> 4);
        const uint32_t d = tmem + x * kTileCols;
        // head dims 16kk .. 16kk+15 in step kk: the half kk/4 of Q and K, 32-byte step kk%4
        tc_mma_ss_k128(d, qt, kt, hi, idesc_s, false);
        tc_commit(&bars->s_full[x]);
        if (last) tc_commit(&bars->q_empty[x]);
      };
      // O_X += P_X V
      auto issue_pv = [&](int x, uint32_t gv, bool acc) {
        const uint32_t vt = v_lo + (((gv % kStages) * kTileBytes) >> 4);
        const uint32_t pt = tmem + x * kTileCols;
        // keys 16kk .. 16kk+15 in step kk: P columns 8kk.., V rows 16kk.. (MN-major)
        static_assert(kKeys == 128 && kHalf == 16384, "the K = 128 issue blocks assume these");
        tc_mma_ts_k128(pt + kOCol, pt, vt, hi, idesc_o, acc);
        tc_commit(&bars->o_done[x]);
      };
      bool ok = true;
      int site = 0, at = 0;
      uint32_t gi = 0, qi[2] = {0, 0}, c[2] = {0, 0}, oi[2] = {0, 0};
      // After a wait on a barrier that other threads' tensor-memory accesses
      // complete (P written, O read) the MMAs that follow are ordered after
      // those accesses with a tcgen05 fence.  Tiles that the TMA loaded need
      // none: the barrier's transaction count already covers the copy.
      auto wait_bar = [&](uint64_t* bar, uint32_t parity, int where, int index,
                          bool tmem_sync) {
        if (!ptx::mbar_wait(bar, parity, kWaitLimit) || *abort_flag) {
          ok = false;
          site = where;
          at = index;
          return false;
        }
        if (tmem_sync) tc_fence_after();
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int w = item_of(k);
        if (w < 0) break;
        const Item it = load_item(dp, w);
        const uint32_t base = gi;
        gi += 2 * it.nmax;
        #pragma unroll
        for (int x = 0; x < 2 && ok; ++x) {
          if (it.n[x] == 0) continue;
          if (wait_bar(&bars->q_full[x], qi[x] & 1, 43, k, false)) ++qi[x];
        }
        // K_0: the first QK^T of both tiles
        if (!ok || !wait_bar(&bars->kv_full[base % kStages], (base / kStages) & 1, 44, (int)base, false))
          break;
        #pragma unroll
        for (int x = 0; x < 2; ++x)
          if (it.n[x] > 0) issue_qk(x, base, it.n[x] == 1);
        tc_commit(&bars->kv_empty[base % kStages]);
        // then per key tile j: PV_A(j) QK_A(j+1) PV_B(j) QK_B(j+1), each tile's
        // products as soon as its softmax has written P
        for (int j = 0; ok && j < it.nmax; ++j) {
          const uint32_t gv = base + 2 * j + 1, gk = gv + 1;
          bool v_in = false, k_in = false;
          #pragma unroll
          for (int x = 0; ok && x < 2; ++x) {
            if (j >= it.n[x]) continue;
            if (!wait_bar(&bars->p_full[x], c[x] & 1, 46, (int)c[x], true)) break;
            if (j == 0 && oi[x] > 0 &&   // the previous item's epilogue must have read O_X
                !wait_bar(&bars->o_free[x], (oi[x] - 1) & 1, 47, (int)oi[x], true))
              break;
            if (!v_in && !wait_bar(&bars->kv_full[gv % kStages], (gv / kStages) & 1, 45, (int)gv, false))
              break;
            v_in = true;
            issue_pv(x, gv, j > 0);
            ++c[x];
            if (j + 1 < it.n[x]) {
              if (!k_in && !wait_bar(&bars->kv_full[gk % kStages], (gk / kStages) & 1, 48, (int)gk, false))
                break;
              k_in = true;
              issue_qk(x, gk, j + 2 == it.n[x]);
            }
          }
          if (!ok) break;
          // a stage is released once every product that reads it was issued
          // (and its copy has landed)
          tc_commit(&bars->kv_empty[gv % kStages]);
          if (j + 1 < it.nmax) {
            if (!k_in && !wait_bar(&bars->kv_full[gk % kStages], (gk / kStages) & 1, 49, (int)gk, false))
              break;
            tc_commit(&bars->kv_empty[gk % kStages]);
          }
        }
        #pragma unroll
        for (int x = 0; x < 2; ++x)
          if (it.n[x] > 0) ++oi[x];
      }
      if (!ok) {
        ptx::report_wait(dp.status, kDevTimeout, site, at);
        *abort_flag = 1;
      }
      // every MMA issued must finish before tensor memory is released
      tc_commit(&bars->drain);
      ptx::mbar_wait(&bars->drain, 0, kWaitLimit);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ------------------------------------------------------------ softmax warps
    const int x = warp >> 2;                          // query tile of this warpgroup
    const int row = threadIdx.x & 127;                // 0..127 = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16) + x * kTileCols;
    const float qk_scale = shp.scale * kLog2e;
    uint32_t cnt = 0, gbase = 0;
    bool ok = true;
    int site = 0, at = 0;
    for (int k = 0; ok; ++k) {
      const int w = item_of(k);
      if (w < 0) break;
      const Item it = load_item(dp, w);
      // this warpgroup's tile, selected without indexing by x (a runtime value)
      const int nx = x ? it.n[1] : it.n[0];
      if (nx == 0) {
        gbase += 2 * it.nmax;
        continue;
      }
      const ChunkTile tile = dp.chunk_tiles[x ? it.tile[1] : it.tile[0]];
      const int h = x ? it.head[1] : it.head[0];
      const int kb = it.kb;
      const int ke = tile.key_end;
      const int pos = tile.pos_begin + row;           // position of this query row
      const uint32_t g_item = gbase;                  // ring index of the item's K_0
      gbase += 2 * it.nmax;
      // keys past the item's end in its last key tile may be anything (unwritten
      // cache slots, and 0 * NaN is NaN): they are zeroed in V, before any PV
      // reads that tile, by A's warpgroup when A reads it (the issuer runs A's
      // PV first), else by B's
      const bool zeroer = (x == 0) ? (nx == it.nmax) : (it.n[0] != it.nmax);
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < nx; ++j) {
        const uint32_t t = cnt + j;
        // tcgen05.ld/st are warp-collective: every decision below is warp-uniform
        const bool got = ptx::mbar_wait(&bars->s_full[x], t & 1, kWaitLimit);
        if (!__all_sync(0xffffffffu, got) || __any_sync(0xffffffffu, *abort_flag != 0)) {
          ok = false;
          site = 51;
          at = (int)t;
          break;
        }
        tc_fence_after();
        const uint32_t s_col = lane_base;               // S of key tile j; then its P
        const int key0 = kb + j * kKeys;
        // this row sees the tile's first `lim` keys: those <= its position and
        // before its tile's end (a prefix of the key tile, possibly empty or all)
        const int lim = min(pos + 1, ke) - key0;
        const bool full = __all_sync(0xffffffffu, lim >= kKeys);
        // the whole row of scores in one round trip (four loads, one wait)
        float sc[128];
        tmem_ld32(s_col, sc);
        tmem_ld32(s_col + 32, sc + 32);
        tmem_ld32(s_col + 64, sc + 64);
        tmem_ld32(s_col + 96, sc + 96);
        tmem_wait_ld();
        if (!full) {
#pragma unroll
          for (int c = 0; c < 128; ++c) sc[c] = c < lim ? sc[c] : -INFINITY;
        }
        // row max: eight independent partial maxima over columns u, u+8, ...,
        // u+120, each built from three-input maxima (half the instructions)
        float mx8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          float a = ptx::fmax3(sc[u], sc[u + 8], sc[u + 16]);
#pragma unroll
          for (int i = 0; i < 6; ++i) a = ptx::fmax3(a, sc[u + 24 + 16 * i], sc[u + 32 + 16 * i]);
          mx8[u] = fmaxf(a, sc[u + 120]);
        }
        const float mraw = ptx::fmax3(ptx::fmax3(mx8[0], mx8[1], mx8[2]),
                                      ptx::fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
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
          const bool done = ptx::mbar_wait(&bars->o_done[x], (t - 1) & 1, kWaitLimit);
          if (!__all_sync(0xffffffffu, done)) {
            ok = false;
            site = 53;
            at = (int)t;
            break;
          }
          tc_fence_after();
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
        // a row with no key in this piece so far keeps m_ref = -inf: its p are 0
        const float nbase = m_ref == -INFINITY ? 0.f : -m_ref;
        // P as bf16 pairs over the first 64 S columns (already read), 64 keys
        // (32 columns) per store.  The scaling and the row sum run as packed
        // pairs (one instruction for two columns): the softmax is bound by
        // instruction issue and the exponentials, and it runs while the
        // tensor pipe works on the other query tile.
        float ps8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) ps8[u] = 0.f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          float pk[32];
          uint32_t* pk32 = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            float x0, x1;
            ptx::fma2(x0, x1, sc[hf * 64 + c], sc[hf * 64 + c + 1], qk_scale, qk_scale, nbase,
                      nbase);
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
        if (zeroer && j == it.nmax - 1 && (it.ke % kKeys) != 0) {
          const uint32_t gv = g_item + 2 * j + 1;     // ring index of V_j
          const int s = gv % kStages;
          const bool landed = ptx::mbar_wait(&bars->kv_full[s], (gv / kStages) & 1, kWaitLimit);
          if (!__all_sync(0xffffffffu, landed)) {
            ok = false;
            site = 52;
            at = (int)gv;
            break;
          }
          uint8_t* vt = kv_s + s * kTileBytes;
          const int valid = it.ke - key0;
          for (int e = row; e < (kKeys - valid) * 16; e += kRows) {
            const int key = valid + e / 16, c = e % 16;
            *reinterpret_cast<uint4*>(vt + (c >> 3) * kHalf + key * 128 + ((c & 7) << 4)) =
                make_uint4(0, 0, 0, 0);
          }
          // the PV MMAs read these rows through the async proxy
          ptx::fence_proxy_async_smem();
        }
        tc_fence_before();
        ptx::mbar_arrive(&bars->p_full[x]);
      }
      if (!ok) break;
      const uint32_t tl = cnt + nx - 1;
      cnt += nx;
      const bool fin = ptx::mbar_wait(&bars->o_done[x], tl & 1, kWaitLimit);
      if (!__all_sync(0xffffffffu, fin)) {
        ok = false;
        site = 54;
        at = (int)tl;
        break;
      }
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool store = row < tile.n_rows;
      const bool partial = tile.part_base >= 0;
      const int kvh = it.kv_head;
      __nv_bfloat16* orow = o + ((int64_t)(tile.row_begin + row) * shp.H_q + h) * 128;
      // partial slot of (row, KV head, split); query head h % g inside it
      const int64_t slot =
          ((int64_t)tile.part_base + ((int64_t)row * shp.H_kv + kvh) * tile.nsplit + tile.split) *
              shp.g + (h % shp.g);
      float* prow = part_o + slot * 128;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float ov[32];
        tmem_ld32(lane_base + kOCol + c4 * 32, ov);
        tmem_wait_ld();
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
      // O_X has been read: the next item's first PV may overwrite it
      tc_fence_before();
      ptx::mbar_arrive(&bars->o_free[x]);
    }
    if (!ok) {
      ptx::report_wait(dp.status, kDevTimeout, site, at);
      *abort_flag = 1;
    }
  }

  // all roles done (every wait above is bounded): release tensor memory
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (!wait_first) ptx::pdl_wait_previous();
}

}  // namespace

bool chunk_fast_supported(const ShapeInfo& s) {
  const bool block_ok = (s.B % kKeys == 0) || (kKeys % s.B == 0 && s.B % 8 == 0);
  return s.dtype == 0 && s.D == 128 && block_ok;
}

cudaError_t launch_chunk_fast(const DevPass& dp, const ShapeInfo& s, const void* q,
                              const void* k_cache, const void* v_cache, void* o, float* part_o,
                              float* part_lse, cudaStream_t st, bool overlap_previous,
                              bool wait_first) {
  if (!chunk_fast_supported(s)) return cudaErrorNotSupported;
  if (dp.n_chunk == 0) return cudaSuccess;
  if (((uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache) & 15)
    return cudaErrorMisalignedAddress;
  if (dp.chunk_single)
    return launch_chunk_single(dp, s, q, k_cache, v_cache, o, part_o, part_lse, st,
                               overlap_previous, wait_first);
  const int64_t rows = (int64_t)dp.num_blocks * s.H_kv * s.B;
  const int box_rows = s.B < kKeys ? s.B : kKeys;
  CUtensorMap tq, tk, tv;
  // Q as [T][H_q * 128]: a query tile is the box at (head * 128, first row),
  // 128 rows high; rows past the end of Q read as zero
  cudaError_t e = make_tmap_2d(&tq, q, dp.num_tokens, (int64_t)s.H_q * 128, kRows);
  if (e == cudaSuccess) e = make_cache_tmap(&tk, k_cache, rows, s.D, box_rows);
  if (e == cudaSuccess) e = make_cache_tmap(&tv, v_cache, rows, s.D, box_rows);
  if (e != cudaSuccess) return e;
  // the shared-memory limit is raised once per device
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t attr_bit = 1ull << (dev & 63);
  if (!(attr_done.load() & attr_bit)) {
    // the register split assumes the kernel was built at kLaunchRegs a thread
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, chunk_attn_tcgen05_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kLaunchRegs) return cudaErrorNotSupported;
    e = cudaFuncSetAttribute(chunk_attn_tcgen05_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(chunk_attn_tcgen05_kernel,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(attr_bit);
  }
  // persistent: at most one CTA per SM, each walking work items
  static int sms_of[64] = {0};
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
  return cudaLaunchKernelEx(&cfg, chunk_attn_tcgen05_kernel, tq, tk, tv, dp, s,
                            (__nv_bfloat16*)o, part_o, part_lse, wait_first ? 1 : 0);
}

}  // namespace rbkv
