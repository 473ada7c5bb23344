// Internal structures shared by the host side (rbkv_host.cpp) and the kernels.
// Nothing here is part of the public ABI (include/rbkv.h).
#pragma once

#include <cuda_runtime_api.h>
#include <stdint.h>

#include "rbkv.h"
#include <nvtx3/nvToolsExt.h>

struct CUtensorMap_st;  // cuda.h's tensor-map type

namespace rbkv {

// A named NVTX range around a library call, so that a profiler that records
// NVTX (`ncu --nvtx`, Nsight Systems) shows composition, appends, attention
// and the layer's steps by name; without such a tool attached the push and
// pop cost a test of a function pointer.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};


// One unit of split attention work: the keys [key_begin, key_end) of one
// sequence's KV head, for n_rows consecutive pass rows of that sequence (all
// query heads of the group each).  Row i of the unit (pass row row + i) sees
// the keys below min(key_end, diag + i): a decode row has n_rows = 1 and
// diag = key_end; a short prompt chunk packs several causal rows.
// part < 0: the unit covers all keys of its rows; write O directly.
// part >= 0 (n_rows = 1 only): write the normalised partial output and its
// log-sum-exp to partial slot `part` of the workspace.
struct WorkItem {
  int32_t row;        // first pass row (index into Q / O)
  int32_t kv_head;
  int32_t key_begin;
  int32_t key_end;
  int32_t part;
  int32_t table_off;  // offset of the sequence's block table in block_ids
  int32_t n_rows;
  int32_t diag;       // keys visible to the unit's first row
};
static_assert(sizeof(WorkItem) == 32, "WorkItem is 8 int32");

// (row, kv head) whose keys were split: partial slots [part_begin, part_begin+nsplit).
struct CombineRow {
  int32_t row;
  int32_t kv_head;
  int32_t part_begin;
  int32_t nsplit;
};

// Up to 128 consecutive rows of one prompt chunk (one sequence), over the keys
// [key_begin, key_end) of one split of their key range.  Row r of the tile is
// pass row row_begin + r at position pos_begin + r; it sees keys
// key_begin .. min(key_end, pos_begin + r + 1) - 1.
// part_base < 0: the tile covers all keys; write O.  Otherwise the partial
// output of row r, KV head k goes to slot part_base + (r * H_kv + k) * nsplit
// + split (each slot holds the g query heads of the KV head).
struct ChunkTile {
  int32_t table_off;
  int32_t row_begin;
  int32_t n_rows;
  int32_t pos_begin;
  int32_t key_begin;
  int32_t key_end;
  int32_t part_base;
  int32_t split;
  int32_t nsplit;
  int32_t pad[3];
};
static_assert(sizeof(ChunkTile) == 48, "ChunkTile is 12 int32");

// Work of one tensor-core CTA step: one or two query tiles that read the same
// K/V tiles - the same rows for two query heads of one KV group, or two
// consecutive 128-row tiles of one chunk for one head (groups of one) - over
// the keys [key_begin, key_end) (the union of the two tiles' key ranges; each
// tile stops at its own key_end).  tile[1] < 0: one query tile.
struct ChunkItem {
  int32_t tile[2];    // indices into the pass's chunk tiles
  int32_t head[2];    // query head of each tile
  int32_t kv_head;
  int32_t key_begin;
  int32_t key_end;
  int32_t pad;
};
static_assert(sizeof(ChunkItem) == 32, "ChunkItem is 8 int32");

// Device view of a pass (pointers into its uploaded metadata buffer).
struct DevPass {
  int32_t* status;                 // device status words (rbkv_status code, wait site, ...)
  const int32_t* slot;             // [T]
  const int32_t* block_ids;        // all block tables
  const WorkItem* decode_items;    // fast decode path
  const WorkItem* generic_items;   // CUDA-core path
  const ChunkTile* chunk_tiles;    // tensor-core prompt path: query tiles
  const ChunkItem* chunk_items;    // ... and the work items over them
  const CombineRow* combine_rows;
  int32_t num_tokens;
  int32_t n_decode;
  int32_t n_generic;
  int32_t n_chunk;                 // chunk work items (ChunkItem)
  int32_t n_combine;
  int32_t n_parts;
  int32_t num_blocks;
  int32_t decode_grid;             // CTAs of the persistent decode launch
  int32_t decode_packed;           // 1: some decode units pack several prompt rows
  int32_t chunk_single;            // 1: chunk items hold one query tile each (the
                                   // one-tile kernel runs them); 0: pairs
  // A frame (rbkv_frame_*): the launches are sized by the frame's capacities
  // (the counts above), and the loaded pass's own counts are read from this
  // device array {num_tokens, n_decode, n_generic, n_chunk (items), n_combine}.
  // Null for a plain pass.
  const int32_t* counts;
};

enum { kCountTokens = 0, kCountDecode = 1, kCountGeneric = 2, kCountChunk = 3, kCountCombine = 4 };

#ifdef __CUDACC__
// The live count `i` of the pass a kernel serves.
__device__ __forceinline__ int32_t pass_count(const DevPass& dp, int i, int32_t fixed) {
  return dp.counts ? dp.counts[i] : fixed;
}
#endif

struct ShapeInfo {
  int32_t H_q, H_kv, D, B, g;
  int32_t dtype;       // rbkv_dtype
  float scale;         // 1/sqrt(D)
};

// Workspace carve-up: partial outputs [n_parts][g][D] fp32, then LSE [n_parts][g].
inline size_t partial_o_bytes(int32_t n_parts, const ShapeInfo& s) {
  size_t b = (size_t)n_parts * s.g * s.D * sizeof(float);
  return (b + 255) / 256 * 256;
}
inline size_t partial_lse_bytes(int32_t n_parts, const ShapeInfo& s) {
  size_t b = (size_t)n_parts * s.g * sizeof(float);
  return (b + 255) / 256 * 256;
}

// Status codes written by kernels (same values as rbkv_status).
constexpr int32_t kDevBounds = -4;
constexpr int32_t kDevTimeout = -7;

// Fast-path envelopes.
constexpr int kDecodeTileKeys = 64;      // keys per pipeline stage of the decode kernel

constexpr int kChunkTileRows = 128;      // query rows per tensor-core tile
constexpr int kChunkTileKeys = 128;      // keys per tensor-core KV tile
constexpr int kChunkMinSplitKeys = 512;  // shortest automatic key split of prompt-chunk tiles
constexpr int kPackedRowsMax = 16;       // prompt chunks of at most this many rows, whose
                                         // keys fit one decode split, go to the decode kernel
constexpr int kDecodeRowsCap = 8;        // query rows x heads of a decode unit, g <= 8

bool decode_fast_supported(const ShapeInfo& s);
// Persistent decode CTAs resident per SM for this shape (1 or 2).
int decode_ctas_per_sm(const ShapeInfo& s);
// 2-D view of a bf16 [num_blocks][H_kv][B][head_dim] cache for TMA: `rows`
// rows of head_dim elements, boxes of 64 columns x box_rows rows, 128 B swizzle.
cudaError_t make_cache_tmap(::CUtensorMap_st* m, const void* cache, int64_t rows,
                            int head_dim, int box_rows);
// Any row-major bf16 [rows][cols] matrix, same box width and swizzle.
cudaError_t make_tmap_2d(::CUtensorMap_st* m, const void* ptr, int64_t rows, int64_t cols,
                         int box_rows);
bool chunk_fast_supported(const ShapeInfo& s);

// Kernel launchers (return the launch's cudaError_t).
cudaError_t launch_kv_append(const DevPass& dp, const ShapeInfo& s, const void* k_new,
                             const void* v_new, void* k_cache, void* v_cache, cudaStream_t st,
                             bool overlap_previous);
// Copy `bytes` (a multiple of 16) of a pass's metadata from mapped pinned
// host memory `src` (a device-accessible address) to device memory `dst`, as a
// kernel that may overlap its predecessor and waits for it before storing.
cudaError_t launch_meta_upload(const void* src, void* dst, size_t bytes, cudaStream_t st,
                               bool overlap_previous);
cudaError_t launch_generic_attention(const DevPass& dp, const ShapeInfo& s, const void* q,
                                     const void* k_cache, const void* v_cache, void* o,
                                     float* part_o, float* part_lse, cudaStream_t st);
// Programmatic dependent launch: overlap_previous lets the kernel start
// before its predecessor in the stream ends; wait_first (decode) makes it
// wait for that predecessor before any global access, for when the
// predecessor is not this call's chunk kernel.
cudaError_t launch_decode_fast(const DevPass& dp, const ShapeInfo& s, const void* q,
                               const void* k_cache, const void* v_cache, void* o,
                               float* part_o, float* part_lse, cudaStream_t st,
                               bool overlap_previous, bool wait_first);
cudaError_t launch_chunk_fast(const DevPass& dp, const ShapeInfo& s, const void* q,
                              const void* k_cache, const void* v_cache, void* o,
                              float* part_o, float* part_lse, cudaStream_t st,
                              bool overlap_previous, bool wait_first);
// The one-tile prompt-chunk kernel (rbkv_chunk_single.cu), for items of one
// query tile each; launch_chunk_fast runs it when dp.chunk_single is set.
cudaError_t launch_chunk_single(const DevPass& dp, const ShapeInfo& s, const void* q,
                                const void* k_cache, const void* v_cache, void* o,
                                float* part_o, float* part_lse, cudaStream_t st,
                                bool overlap_previous, bool wait_first);
cudaError_t launch_combine(const DevPass& dp, const ShapeInfo& s, const float* part_o,
                           const float* part_lse, void* o, cudaStream_t st);
// Decoder-layer dense steps (rbkv_gemm.cu): C = A B^T with an epilogue
// (0 plain, 1 + residual, 2 SwiGLU over 128-row gate/up blocks of B, 3 C's
// columns split at split1 and split2 into c, c2 and c3; ldc is C's row
// stride), and RMSNorm of M rows of H.
cudaError_t launch_gemm_bf16(const void* a, const void* b, void* c, const void* r, int64_t M,
                             int64_t N, int64_t K, int64_t ldc, int epilogue, int32_t* status,
                             cudaStream_t st, void* c2 = nullptr, void* c3 = nullptr,
                             int64_t split1 = 0, int64_t split2 = 0, void* ws = nullptr,
                             size_t ws_bytes = 0);
// Workspace a GEMM of this size uses to split K (0: it does not split).
size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_rmsnorm_bf16(const void* x, const void* w, void* y, int64_t M, int64_t H,
                                float eps, cudaStream_t st);
// One CTA waiting `limit` cycles on a barrier nothing completes; reports the
// timeout in `status` (diagnostics).
cudaError_t launch_wait_timeout(int32_t* status, long long limit, cudaStream_t st);

// Host helpers for the entry point that allocates nothing (rbkv_noalloc.cu).
// attention_on_device: rbkv_ragged_attention for a pass whose metadata is
// already on the current device, with `scratch` as its workspace; it never
// allocates.  set_error: record a message for rbkv_last_error.
rbkv_status attention_on_device(rbkv_pass* p, const void* q, const void* k_cache,
                                const void* v_cache, void* o, void* scratch,
                                size_t scratch_bytes, cudaStream_t st);
rbkv_status set_error(rbkv_status st, const char* msg);
// Count n kernel launches made outside rbkv_host.cpp (rbkv_kernel_launches).
void note_launches(int64_t n);
}  // namespace rbkv
