// Host side of librbkv: the Dynamic SplitFuse composer, the block pool, the
// split-KV planner, the metadata packer and the C ABI entry points.
//
// Composition follows the DeepSpeed-FastGen paper summary page ("Summary",
// idea I3): a pass holds a fixed token budget; long prompts are chunked over
// passes; generation tokens and short prompts top the pass up.  Split planning
// follows the FastGen guide ("Dynamic SplitKV Attention"): the number of key
// splits of a decode row grows with its context so that every SM has work.
#include "rbkv.h"
#include "rbkv_internal.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <mutex>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

using namespace rbkv;

namespace {

thread_local std::string g_err;

rbkv_status fail(rbkv_status st, const std::string& msg) {
  g_err = msg;
  return st;
}

rbkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(RBKV_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

constexpr int32_t kMaxTokens = 1 << 30;

// ---- block pool: one bit per block, set = free; lowest free id first --------
class BlockPool {
 public:
  explicit BlockPool(int32_t n) : n_(n), nfree_(n), hint_(0) {
    words_.assign((size_t)(n + 63) / 64, ~0ull);
    if (n % 64) words_.back() = (1ull << (n % 64)) - 1;
    if (n == 0) words_.clear();
  }
  int32_t free_count() const { return nfree_; }
  int32_t take_lowest() {
    for (size_t w = hint_; w < words_.size(); ++w) {
      if (words_[w]) {
        int bit = __builtin_ctzll(words_[w]);
        words_[w] &= ~(1ull << bit);
        hint_ = w;
        --nfree_;
        return (int32_t)(w * 64 + bit);
      }
    }
    return -1;
  }
  void give_back(int32_t b) {
    words_[(size_t)b / 64] |= 1ull << (b % 64);
    hint_ = std::min(hint_, (size_t)b / 64);
    ++nfree_;
  }

 private:
  std::vector<uint64_t> words_;
  int32_t n_, nfree_;
  size_t hint_;
};

// ---- pinned staging buffers for the per-pass metadata upload ---------------
// Mapped pinned host memory: the upload kernel reads it directly.  A buffer
// goes back to the pool as soon as its upload is enqueued; it is reused only
// once the event recorded after that upload has completed.
struct PinnedBuf {
  void* ptr = nullptr;
  void* dptr = nullptr;   // the same memory's device-accessible address (mapped)
  size_t cap = 0;
  cudaEvent_t ev = nullptr;
};

class PinnedPool {
 public:
  ~PinnedPool() {
    for (auto& b : free_) {
      if (b.ev) { cudaEventSynchronize(b.ev); cudaEventDestroy(b.ev); }
      if (b.ptr) cudaFreeHost(b.ptr);
    }
  }
  cudaError_t acquire(size_t bytes, PinnedBuf& out) {
    for (size_t i = 0; i < free_.size(); ++i) {
      if (free_[i].cap >= bytes && cudaEventQuery(free_[i].ev) == cudaSuccess) {
        out = free_[i];
        free_.erase(free_.begin() + i);
        return cudaSuccess;
      }
    }
    (void)cudaGetLastError();  // cudaEventQuery may have left cudaErrorNotReady
    size_t cap = 4096;
    while (cap < bytes) cap *= 2;
    PinnedBuf b;
    cudaError_t e = cudaHostAlloc(&b.ptr, cap, cudaHostAllocMapped);
    if (e != cudaSuccess) return e;
    e = cudaHostGetDevicePointer(&b.dptr, b.ptr, 0);
    if (e != cudaSuccess) { cudaFreeHost(b.ptr); return e; }
    e = cudaEventCreateWithFlags(&b.ev, cudaEventDisableTiming);
    if (e != cudaSuccess) { cudaFreeHost(b.ptr); return e; }
    b.cap = cap;
    out = b;
    return cudaSuccess;
  }
  void release(const PinnedBuf& b) {
    free_.push_back(b);
    if (free_.size() > 64) {  // keep the pool small: drop the oldest idle buffer
      PinnedBuf old = free_.front();
      cudaEventSynchronize(old.ev);
      cudaEventDestroy(old.ev);
      cudaFreeHost(old.ptr);
      free_.erase(free_.begin());
    }
  }

 private:
  std::vector<PinnedBuf> free_;
};

// ---- launch counting and optional per-launch event timing -------------------
std::atomic<int64_t> g_launches{0};

struct Profiler {
  bool on = false;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> rec[RBKV_KERNEL_KINDS];
  std::vector<cudaEvent_t> spare;
  cudaEvent_t get() {
    cudaEvent_t e = nullptr;
    if (!spare.empty()) { e = spare.back(); spare.pop_back(); return e; }
    cudaEventCreate(&e);
    return e;
  }
  void reset() {
    for (auto& r : rec) {
      for (auto& pr : r) { spare.push_back(pr.first); spare.push_back(pr.second); }
      r.clear();
    }
  }
};
Profiler g_prof;

template <class F>
cudaError_t launch_counted(int kind, cudaStream_t st, F&& f) {
  cudaEvent_t a = nullptr;
  if (g_prof.on) { a = g_prof.get(); cudaEventRecord(a, st); }
  cudaError_t e = f();
  if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
  if (g_prof.on) {
    cudaEvent_t b = g_prof.get();
    cudaEventRecord(b, st);
    g_prof.rec[kind].push_back({a, b});
  }
  return e;
}

int32_t ceil_div(int64_t a, int64_t b) { return (int32_t)((a + b - 1) / b); }
int32_t round_up(int64_t a, int64_t b) { return (int32_t)((a + b - 1) / b * b); }

// ---- the attention plan of one pass -----------------------------------------
struct Plan {
  rbkv_plan_info info{};
  std::vector<WorkItem> decode, generic;
  std::vector<ChunkTile> chunk;
  std::vector<ChunkItem> chunk_items;
  std::vector<CombineRow> combine;
  int64_t chunk_steps_total = 0, chunk_steps_max = 0;
  int64_t decode_keys_total = 0, decode_keys_max = 0;
  int32_t n_parts = 0;
  int32_t decode_grid = 0;
  int32_t decode_packed = 0;  // some decode units pack several prompt rows
  int32_t chunk_single = 0;   // chunk items hold one query tile each
};

}  // namespace

struct rbkv_composer {
  rbkv_config cfg;
  BlockPool pool;
  std::unordered_map<int64_t, std::vector<int32_t>> held;
  std::unordered_map<int64_t, int32_t> tokens;
  std::shared_ptr<PinnedPool> pinned;
  explicit rbkv_composer(const rbkv_config& c)
      : cfg(c), pool(c.num_blocks), pinned(std::make_shared<PinnedPool>()) {}
};

struct rbkv_pass {
  rbkv_config cfg;
  std::shared_ptr<PinnedPool> pinned;
  std::vector<int64_t> seq_ids;
  std::vector<int32_t> q_start{0}, n_new, seen, ctx, block_start{0}, block_ids, slot;
  int32_t split_keys = 0;
  int32_t chunk_items = RBKV_CHUNK_ITEMS_AUTO;
  // plan, made once for the device of the first device call
  bool planned = false;
  int device = -1;
  Plan plan;
  // device copy of the metadata
  void* dev = nullptr;
  size_t dev_bytes = 0;
  cudaStream_t upload_stream = nullptr;
  cudaStream_t last_stream = nullptr;
  std::vector<cudaStream_t> streams;   // every stream device work of the pass was put on
  cudaEvent_t upload_ev = nullptr;
  DevPass dp{};
  void use_stream(cudaStream_t st) {
    last_stream = st;
    if (std::find(streams.begin(), streams.end(), st) == streams.end()) streams.push_back(st);
  }
};

namespace {

ShapeInfo shape_of(const rbkv_config& c) {
  ShapeInfo s;
  s.H_q = c.num_heads_q;
  s.H_kv = c.num_heads_kv;
  s.D = c.head_dim;
  s.B = c.block_size;
  s.g = c.num_heads_q / c.num_heads_kv;
  s.dtype = c.dtype;
  s.scale = (float)(1.0 / std::sqrt((double)c.head_dim));
  return s;
}

// Split the keys [0, n_keys) of one (row, kv head) into near-equal pieces of
// at most `split` keys, each a multiple of `gran` except the last.
void split_keys(int32_t n_keys, int32_t split, int32_t gran, std::vector<int32_t>& bounds) {
  bounds.clear();
  int32_t nsplit = std::max(1, ceil_div(n_keys, split));
  int32_t piece = round_up(ceil_div(n_keys, nsplit), gran);
  for (int32_t k = 0; k < n_keys; k += piece) bounds.push_back(k);
  bounds.push_back(n_keys);
}

// The snake deal of decode units is refined when there are at most this many
// per CTA (more of them even out under the snake deal alone), a unit costing
// its keys plus this many for its start-up and merge (about 0.7 us of a CTA
// streaming about 45 keys a microsecond).
constexpr int32_t kDecodeBalanceUnits = 4;
constexpr int32_t kDecodeUnitStartKeys = 32;

// Reorder `items` (sorted longest first) so that a persistent grid of G CTAs,
// CTA c taking items c, c+G, c+2G, ..., receives them in snake order: round r
// hands sorted items r*G .. r*G+G-1 to CTAs 0..G-1 on even rounds and to
// G-1..0 on odd rounds.  Long and short units even out across CTAs.
void snake_order(std::vector<WorkItem>& items, int32_t G) {
  std::vector<WorkItem> out(items.size());
  for (size_t i = 0; i < items.size(); ++i) {
    size_t r = i / G, c = i % G;
    size_t base = r * G;
    size_t width = std::min((size_t)G, items.size() - base);
    size_t src = (r % 2 == 0) ? base + c : base + (width - 1 - c);
    out[i] = items[src];
  }
  items.swap(out);
}

// Even out the work of a persistent grid of G CTAs in which CTA cta_of(pos)
// walks position `pos` of `items`.  The given placement is the start (snake
// dealing of items sorted longest first leaves the CTAs of a last, partial
// round one item above the rest, and with few items per CTA the busiest about
// a tenth above the mean); items are then swapped one for one (so every CTA
// keeps its number of positions) between the most and the least loaded CTA
// while a swap narrows their gap, and each CTA takes its items costliest
// first.  `cost[pos]` is the work of the item at `pos`; returns the most work
// one CTA gets.  A few flat arrays, no allocation per CTA: the planner runs
// for every pass.
template <class T, class CtaOf>
int64_t balance_items(std::vector<T>& items, int32_t G, const std::vector<int32_t>& cost,
                      CtaOf cta_of) {
  const size_t n = items.size();
  if (G <= 0 || n <= (size_t)G)
    return n ? (int64_t)*std::max_element(cost.begin(), cost.end()) : 0;
  // slot[start[b] ..] = the items of CTA b (indices into `items`)
  std::vector<int32_t> start(G + 1, 0), fill(G, 0), slot(n);
  std::vector<int64_t> load(G, 0);
  for (size_t pos = 0; pos < n; ++pos) ++start[cta_of(pos) + 1];
  for (int32_t b = 0; b < G; ++b) start[b + 1] += start[b];
  for (size_t pos = 0; pos < n; ++pos) {
    const int32_t b = cta_of(pos);
    slot[start[b] + fill[b]++] = (int32_t)pos;
    load[b] += cost[pos];
  }
  // the most and the least loaded CTA (ties: lowest index) from two heaps of
  // (load, CTA) entries; an entry whose load is no longer the CTA's is stale
  // and dropped when it comes to the top
  using Entry = std::pair<int64_t, int32_t>;
  std::vector<Entry> most, least;   // keys (load, -b) and (load, b)
  most.reserve(G + 256);
  least.reserve(G + 256);
  const auto greater = [](const Entry& x, const Entry& y) { return x > y; };
  for (int32_t b = 0; b < G; ++b) {
    most.push_back({load[b], -b});
    least.push_back({load[b], b});
  }
  std::make_heap(most.begin(), most.end());
  std::make_heap(least.begin(), least.end(), greater);
  auto top_most = [&]() {
    while (load[-most.front().second] != most.front().first) {
      std::pop_heap(most.begin(), most.end());
      most.pop_back();
    }
    return -most.front().second;
  };
  auto top_least = [&]() {
    while (load[least.front().second] != least.front().first) {
      std::pop_heap(least.begin(), least.end(), greater);
      least.pop_back();
    }
    return least.front().second;
  };
  for (int iter = 0; iter < 8 * G; ++iter) {
    const int32_t hi = top_most(), lo = top_least();
    const int64_t gap = load[hi] - load[lo];
    int32_t best_a = -1, best_b = -1;
    int64_t best_d = 0;
    for (int32_t a = start[hi]; a < start[hi + 1]; ++a)
      for (int32_t c = start[lo]; c < start[lo + 1]; ++c) {
        const int64_t d = (int64_t)cost[slot[a]] - cost[slot[c]];
        if (d <= 0 || d >= gap) continue;
        if (best_a < 0 || std::llabs(gap - 2 * d) < std::llabs(gap - 2 * best_d)) {
          best_a = a;
          best_b = c;
          best_d = d;
        }
      }
    if (best_a < 0) break;
    std::swap(slot[best_a], slot[best_b]);
    load[hi] -= best_d;
    load[lo] += best_d;
    for (const int32_t b : {hi, lo}) {
      most.push_back({load[b], -b});
      std::push_heap(most.begin(), most.end());
      least.push_back({load[b], b});
      std::push_heap(least.begin(), least.end(), greater);
    }
  }
  // each CTA's items costliest first (insertion sort: a few items each;
  // equal costs keep their order)
  for (int32_t b = 0; b < G; ++b)
    for (int32_t i = start[b] + 1; i < start[b + 1]; ++i) {
      const int32_t v = slot[i];
      int32_t j = i;
      for (; j > start[b] && cost[slot[j - 1]] < cost[v]; --j) slot[j] = slot[j - 1];
      slot[j] = v;
    }
  std::vector<T> out(n);
  std::fill(fill.begin(), fill.end(), 0);
  for (size_t pos = 0; pos < n; ++pos) {
    const int32_t b = cta_of(pos);
    out[pos] = items[slot[start[b] + fill[b]++]];
  }
  items.swap(out);
  return *std::max_element(load.begin(), load.end());
}

Plan make_plan(const rbkv_pass& p, int32_t num_sms) {
  Plan pl;
  ShapeInfo s = shape_of(p.cfg);
  const bool fast_decode = decode_fast_supported(s);
  const bool fast_chunk = chunk_fast_supported(s);
  const int32_t gran = fast_decode ? kDecodeTileKeys : 16;
  const int32_t S = (int32_t)p.seq_ids.size();

  int64_t decode_work = 0;
  int32_t decode_rows = 0, chunk_rows = 0;
  for (int32_t i = 0; i < S; ++i) {
    if (p.n_new[i] == 1) { decode_work += (int64_t)p.ctx[i] * s.H_kv; ++decode_rows; }
    else chunk_rows += p.n_new[i];
  }
  int32_t split;
  if (p.split_keys > 0) {
    split = round_up(p.split_keys, gran);
  } else {
    // about four units per SM of equal size, never shorter than 512 keys
    // (every unit costs a start-up, a merge and, when split, a partial output
    // and its combine: shorter units cost more than they gain in balance)
    int64_t slots = (int64_t)std::max(1, num_sms);
    int64_t target = (decode_work + slots * 4 - 1) / (slots * 4);
    split = std::max<int32_t>(512, round_up(std::max<int64_t>(target, 1), gran));
  }

  // prompt chunks: 128-row query tiles in work items.  When there are at
  // least as many pairs of tiles that read the same K/V tiles (two query heads
  // of a KV group, or two consecutive row tiles for groups of one) as SMs,
  // items are such pairs (the paired kernel overlaps one tile's softmax with
  // the other's products); otherwise items hold one tile and query head each
  // (the one-tile kernel, whose double-buffered scores overlap each tile's
  // softmax with its own next product), and a chunk's key range is split only
  // when even those are fewer than SMs, into pieces that bring the count up to
  // about one full wave.  The persistent grid has one CTA per SM.
  int32_t chunk_split = 0x7fffffff;
  bool chunk_single = false;
  if (fast_chunk) {
    int64_t pairs = 0, singles = 0;
    int32_t max_keys = 0;
    for (int32_t i = 0; i < S; ++i) {
      if (p.n_new[i] <= 1) continue;
      const int64_t tiles = ceil_div(p.n_new[i], kChunkTileRows);
      pairs += s.g >= 2 ? tiles * s.H_kv * ceil_div(s.g, 2) : ceil_div(tiles, 2) * s.H_q;
      singles += tiles * s.H_q;
      max_keys = std::max(max_keys, p.ctx[i]);
    }
    chunk_single = p.chunk_items == RBKV_CHUNK_ITEMS_AUTO ? pairs < num_sms
                                                          : p.chunk_items == RBKV_CHUNK_ITEMS_SINGLE;
    if (p.split_keys > 0) {
      chunk_split = round_up(p.split_keys, kChunkTileKeys);
    } else if (singles > 0 && singles < num_sms) {
      const int32_t per = std::max<int32_t>(1, (int32_t)(num_sms / singles));
      chunk_split = std::max<int32_t>(kChunkMinSplitKeys,
                                      round_up(ceil_div(max_keys, per), kChunkTileKeys));
    }
  }
  pl.chunk_single = chunk_single ? 1 : 0;
  std::vector<int32_t> bounds;
  std::vector<WorkItem> decode, generic;
  int32_t max_splits = 0;
  // Decode-kernel work is planned per row first: the key split of a row is the
  // same for all its KV heads, so a row's pieces (one per key split, or one per
  // packed group of prompt rows) are made and sorted longest first, and only
  // then expanded into one unit per KV head.  Partial slot of (row, head h,
  // split k): part0 + h * nsplit + k.
  struct Piece {
    int32_t row, key_begin, key_end, part0, k, nsplit, table_off, n_rows, diag;
  };
  std::vector<Piece> pieces;
  pieces.reserve((size_t)S * 2);
  std::vector<int32_t> tile_of;   // chunk tile of (row tile, key piece), or -1
  auto add_decode_row = [&](int32_t row, int32_t n_keys, int32_t table_off) {
    split_keys(n_keys, split, gran, bounds);
    const int32_t ns = (int32_t)bounds.size() - 1;
    max_splits = std::max(max_splits, ns);
    int32_t part0 = -1;
    if (ns > 1) {
      part0 = pl.n_parts;
      pl.n_parts += ns * s.H_kv;
      for (int32_t h = 0; h < s.H_kv; ++h)
        pl.combine.push_back(CombineRow{row, h, part0 + h * ns, ns});
    }
    for (int32_t k = 0; k < ns; ++k)
      pieces.push_back(Piece{row, bounds[k], bounds[k + 1], part0, k, ns, table_off, 1, n_keys});
  };
  // CUDA-core units: (row, kv head, split), as before
  auto add_generic_row = [&](int32_t row, int32_t n_keys, int32_t table_off) {
    for (int32_t h = 0; h < s.H_kv; ++h) {
      split_keys(n_keys, split, gran, bounds);
      int32_t ns = (int32_t)bounds.size() - 1;
      max_splits = std::max(max_splits, ns);
      int32_t part0 = -1;
      if (ns > 1) {
        part0 = pl.n_parts;
        pl.n_parts += ns;
        pl.combine.push_back(CombineRow{row, h, part0, ns});
      }
      for (int32_t k = 0; k < ns; ++k)
        generic.push_back(WorkItem{row, h, bounds[k], bounds[k + 1], ns > 1 ? part0 + k : -1,
                                   table_off, 1, n_keys});
    }
  };
  // rows of a short prompt chunk per decode unit: all g query heads of each
  const int32_t pack = s.g <= kDecodeRowsCap ? kDecodeRowsCap / s.g : 1;
  for (int32_t i = 0; i < S; ++i) {
    if (p.n_new[i] == 1) {
      if (fast_decode) add_decode_row(p.q_start[i], p.ctx[i], p.block_start[i]);
      else add_generic_row(p.q_start[i], p.ctx[i], p.block_start[i]);
    } else if (fast_decode && p.n_new[i] <= kPackedRowsMax && p.ctx[i] <= split) {
      // a short prompt chunk whose keys fit one decode unit: causal rows packed
      // `pack` at a time into decode units (no tensor-core tile of 128 rows)
      for (int32_t j = 0; j < p.n_new[i]; j += pack) {
        const int32_t n = std::min(pack, p.n_new[i] - j);
        pieces.push_back(Piece{p.q_start[i] + j, 0, p.seen[i] + j + n, -1, 0, 1,
                               p.block_start[i], n, p.seen[i] + j + 1});
      }
      max_splits = std::max(max_splits, 1);
      pl.decode_packed = 1;
    } else if (fast_chunk) {
      // the chunk's keys [0, ctx) are cut into 128-key-aligned pieces of at
      // most `chunk_split` keys; 128-row tile t takes from piece k the keys
      // below its own causal end (pieces that start past it are left out), and
      // a tile with several pieces has them merged by the log-sum-exp combine
      split_keys(p.ctx[i], chunk_split, kChunkTileKeys, bounds);
      const int32_t npiece = (int32_t)bounds.size() - 1;
      const int32_t ntile = ceil_div(p.n_new[i], kChunkTileRows);
      tile_of.assign((size_t)ntile * npiece, -1);
      for (int32_t t = 0; t < ntile; ++t) {
        const int32_t r = t * kChunkTileRows;
        const int32_t n = std::min(kChunkTileRows, p.n_new[i] - r);
        const int32_t pos0 = p.seen[i] + r;
        const int32_t tile_end = pos0 + n;
        int32_t ns = 0;
        while (ns < npiece && bounds[ns] < tile_end) ++ns;
        max_splits = std::max(max_splits, ns);
        int32_t part0 = -1;
        if (ns > 1) {
          part0 = pl.n_parts;
          pl.n_parts += n * s.H_kv * ns;
          for (int32_t rr = 0; rr < n; ++rr)
            for (int32_t h = 0; h < s.H_kv; ++h)
              pl.combine.push_back(
                  CombineRow{p.q_start[i] + r + rr, h, part0 + (rr * s.H_kv + h) * ns, ns});
        }
        for (int32_t k = 0; k < ns; ++k) {
          tile_of[(size_t)t * npiece + k] = (int32_t)pl.chunk.size();
          pl.chunk.push_back(ChunkTile{p.block_start[i], p.q_start[i] + r, n, pos0, bounds[k],
                                       std::min(bounds[k + 1], tile_end), part0, k, ns,
                                       {0, 0, 0}});
        }
      }
      auto key_end_of = [&](int32_t a, int32_t b) {
        const int32_t ea = a >= 0 ? pl.chunk[a].key_end : 0;
        const int32_t eb = b >= 0 ? pl.chunk[b].key_end : 0;
        return std::max(ea, eb);
      };
      for (int32_t k = 0; k < npiece; ++k) {
        if (chunk_single) {
          // one tile and query head per item
          for (int32_t t = 0; t < ntile; ++t) {
            const int32_t c = tile_of[(size_t)t * npiece + k];
            if (c < 0) continue;
            for (int32_t h = 0; h < s.H_q; ++h)
              pl.chunk_items.push_back(ChunkItem{{c, -1}, {h, 0}, h / s.g,
                                                 pl.chunk[c].key_begin, pl.chunk[c].key_end, 0});
          }
        } else if (s.g >= 2) {
          // each tile with two query heads of a KV group per item
          for (int32_t t = 0; t < ntile; ++t) {
            const int32_t c = tile_of[(size_t)t * npiece + k];
            if (c < 0) continue;
            for (int32_t h = 0; h < s.H_kv; ++h)
              for (int32_t q = 0; q < s.g; q += 2) {
                const bool two = q + 1 < s.g;
                pl.chunk_items.push_back(ChunkItem{{c, two ? c : -1},
                                                   {h * s.g + q, two ? h * s.g + q + 1 : 0}, h,
                                                   pl.chunk[c].key_begin, pl.chunk[c].key_end,
                                                   0});
              }
          }
        } else {
          // groups of one: two consecutive row tiles of one head per item
          for (int32_t t = 0; t < ntile; t += 2) {
            int32_t a = tile_of[(size_t)t * npiece + k];
            int32_t b = t + 1 < ntile ? tile_of[(size_t)(t + 1) * npiece + k] : -1;
            if (a < 0) { a = b; b = -1; }
            if (a < 0) continue;
            for (int32_t h = 0; h < s.H_q; ++h)
              pl.chunk_items.push_back(ChunkItem{{a, b}, {h, h}, h, bounds[k], key_end_of(a, b),
                                                 0});
          }
        }
      }
    } else {
      for (int32_t j = 0; j < p.n_new[i]; ++j)
        add_generic_row(p.q_start[i] + j, p.seen[i] + j + 1, p.block_start[i]);
    }
  }
  std::stable_sort(pieces.begin(), pieces.end(), [](const Piece& a, const Piece& b) {
    return (a.key_end - a.key_begin) > (b.key_end - b.key_begin);
  });
  decode.reserve(pieces.size() * (size_t)s.H_kv);
  for (const Piece& pc : pieces)
    for (int32_t h = 0; h < s.H_kv; ++h)
      decode.push_back(WorkItem{pc.row, h, pc.key_begin, pc.key_end,
                                pc.part0 >= 0 ? pc.part0 + h * pc.nsplit + pc.k : -1,
                                pc.table_off, pc.n_rows, pc.diag});
  auto longer = [](const WorkItem& a, const WorkItem& b) {
    return (a.key_end - a.key_begin) > (b.key_end - b.key_begin);
  };
  std::stable_sort(generic.begin(), generic.end(), longer);
  std::stable_sort(pl.chunk_items.begin(), pl.chunk_items.end(),
                   [](const ChunkItem& a, const ChunkItem& b) {
                     return (a.key_end - a.key_begin) > (b.key_end - b.key_begin);
                   });
  if (!pl.chunk_items.empty()) {
    // an item's work: the key-tile steps of its query tiles, plus one for its
    // epilogue
    std::vector<int32_t> cost(pl.chunk_items.size());
    for (size_t i = 0; i < cost.size(); ++i) {
      const ChunkItem& ci = pl.chunk_items[i];
      int32_t c = 1;
      for (int x = 0; x < 2; ++x)
        if (ci.tile[x] >= 0)
          c += ceil_div(pl.chunk[ci.tile[x]].key_end - ci.key_begin, kChunkTileKeys);
      cost[i] = c;
    }
    for (int32_t c : cost) pl.chunk_steps_total += c;
    // the chunk grid walks its positions in snake order: CTA b takes, in
    // round k, position k*G + b on even rounds and k*G + G-1-b on odd ones
    const int32_t G = (int32_t)std::min<int64_t>((int64_t)cost.size(), std::max(1, num_sms));
    pl.chunk_steps_max = balance_items(pl.chunk_items, G, cost, [G](size_t pos) -> int32_t {
      const size_t k = pos / G, i = pos % G;
      return (int32_t)((k & 1) ? G - 1 - i : i);
    });
  }
  int32_t grid =(int32_t)std::min<int64_t>((int64_t)decode.size(),
                                            (int64_t)std::max(1, num_sms) * decode_ctas_per_sm(s));
  if (grid > 0) {
    // the decode grid walks positions c, c + G, c + 2G, ... (CTA c); the
    // snake deal is the placement, refined when there are few units per CTA
    snake_order(decode, grid);
    if (decode.size() <= (size_t)kDecodeBalanceUnits * grid) {
      std::vector<int32_t> cost(decode.size());
      for (size_t i = 0; i < decode.size(); ++i)
        cost[i] = decode[i].key_end - decode[i].key_begin + kDecodeUnitStartKeys;
      balance_items(decode, grid, cost, [grid](size_t pos) { return (int32_t)(pos % grid); });
    }
    std::vector<int64_t> keys(grid, 0);
    for (size_t i = 0; i < decode.size(); ++i) {
      const int64_t k = decode[i].key_end - decode[i].key_begin;
      keys[i % grid] += k;
      pl.decode_keys_total += k;
    }
    pl.decode_keys_max = *std::max_element(keys.begin(), keys.end());
  }
  pl.decode_grid = grid;
  pl.decode.swap(decode);
  pl.generic.swap(generic);

  rbkv_plan_info& in = pl.info;
  in.num_sms = num_sms;
  in.decode_rows = decode_rows;
  in.decode_items = fast_decode ? (int32_t)pl.decode.size() : 0;
  in.max_splits = max_splits;
  in.split_keys = split;
  in.partials = pl.n_parts;
  in.chunk_rows = chunk_rows;
  in.chunk_tiles = (int32_t)pl.chunk.size();
  in.chunk_items = (int32_t)pl.chunk_items.size();
  in.chunk_single = pl.chunk_single;
  in.chunk_steps_total = (int32_t)std::min<int64_t>(pl.chunk_steps_total, INT32_MAX);
  in.chunk_steps_max = (int32_t)std::min<int64_t>(pl.chunk_steps_max, INT32_MAX);
  in.decode_grid = pl.decode_grid;
  in.decode_keys_total = (int32_t)std::min<int64_t>(pl.decode_keys_total, INT32_MAX);
  in.decode_keys_max = (int32_t)std::min<int64_t>(pl.decode_keys_max, INT32_MAX);
  in.generic_items = (int32_t)pl.generic.size();
  in.fast_decode = fast_decode ? 1 : 0;
  in.fast_chunk = fast_chunk ? 1 : 0;
  return pl;
}

size_t workspace_bytes_of(const rbkv_pass& p) {
  if (p.plan.n_parts == 0) return 0;
  ShapeInfo s = shape_of(p.cfg);
  return partial_o_bytes(p.plan.n_parts, s) + partial_lse_bytes(p.plan.n_parts, s);
}

rbkv_status ensure_plan(rbkv_pass* p) {
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (p->planned) {
    if (dev != p->device)
      return fail(RBKV_ERR_INVALID, "pass was bound to another device by its first device call");
    return RBKV_OK;
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  p->plan = make_plan(*p, sms);
  p->device = dev;
  p->planned = true;
  return RBKV_OK;
}


// Plan (if needed), pack and upload the metadata on `st`; order `st` after
// the upload when it is another stream.
rbkv_status ensure_device(rbkv_pass* p, cudaStream_t st) {
  rbkv_status rs = ensure_plan(p);
  if (rs != RBKV_OK) return rs;
  if (!p->dev) {
    const Plan& pl = p->plan;
    // sections of int32 words, each 16-byte aligned, after four status words:
    // packed straight into pinned staging memory
    size_t words = 4;
    auto section = [&words](size_t bytes) {
      const size_t off = words;
      words = (words + bytes / 4 + 3) / 4 * 4;
      return off;
    };
    const size_t o_slot = section(p->slot.size() * 4);
    const size_t o_blocks = section(p->block_ids.size() * 4);
    const size_t o_dec = section(pl.decode.size() * sizeof(WorkItem));
    const size_t o_gen = section(pl.generic.size() * sizeof(WorkItem));
    const size_t o_chunk = section(pl.chunk.size() * sizeof(ChunkTile));
    const size_t o_items = section(pl.chunk_items.size() * sizeof(ChunkItem));
    const size_t o_comb = section(pl.combine.size() * sizeof(CombineRow));
    const size_t bytes = words * 4;
    PinnedBuf pin;
    cudaError_t e = p->pinned->acquire(bytes, pin);
    if (e != cudaSuccess) return cuda_fail(e, "cudaHostAlloc");
    int32_t* hw = (int32_t*)pin.ptr;
    std::memset(hw, 0, 16);   // status words: code, wait site, index, block
    auto fill = [hw](size_t off, const void* src, size_t n) {
      if (n) std::memcpy(hw + off, src, n);
    };
    fill(o_slot, p->slot.data(), p->slot.size() * 4);
    fill(o_blocks, p->block_ids.data(), p->block_ids.size() * 4);
    fill(o_dec, pl.decode.data(), pl.decode.size() * sizeof(WorkItem));
    fill(o_gen, pl.generic.data(), pl.generic.size() * sizeof(WorkItem));
    fill(o_chunk, pl.chunk.data(), pl.chunk.size() * sizeof(ChunkTile));
    fill(o_items, pl.chunk_items.data(), pl.chunk_items.size() * sizeof(ChunkItem));
    fill(o_comb, pl.combine.data(), pl.combine.size() * sizeof(CombineRow));
    void* dev = nullptr;
    e = cudaMallocAsync(&dev, bytes, st);
    if (e != cudaSuccess) { p->pinned->release(pin); return cuda_fail(e, "cudaMallocAsync"); }
    // the upload is the pass's first kernel: it overlaps the previous kernel
    // in the stream and stores only after that kernel has finished
    e = launch_counted(RBKV_KERNEL_META_UPLOAD, st, [&] {
      return launch_meta_upload(pin.dptr, dev, bytes, st, !g_prof.on);
    });
    if (e == cudaSuccess) e = cudaEventRecord(pin.ev, st);
    p->pinned->release(pin);
    if (e != cudaSuccess) { cudaFreeAsync(dev, st); return cuda_fail(e, "metadata upload"); }
    e = cudaEventCreateWithFlags(&p->upload_ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(p->upload_ev, st);
    if (e != cudaSuccess) { cudaFreeAsync(dev, st); return cuda_fail(e, "upload event"); }
    p->dev = dev;
    p->dev_bytes = bytes;
    p->upload_stream = st;
    int32_t* base = (int32_t*)dev;
    DevPass& dp = p->dp;
    dp.status = base;
    dp.slot = base + o_slot;
    dp.block_ids = base + o_blocks;
    dp.decode_items = (const WorkItem*)(base + o_dec);
    dp.generic_items = (const WorkItem*)(base + o_gen);
    dp.chunk_tiles = (const ChunkTile*)(base + o_chunk);
    dp.chunk_items = (const ChunkItem*)(base + o_items);
    dp.combine_rows = (const CombineRow*)(base + o_comb);
    dp.num_tokens = (int32_t)p->slot.size();
    dp.n_decode = (int32_t)pl.decode.size();
    dp.n_generic = (int32_t)pl.generic.size();
    dp.n_chunk = (int32_t)pl.chunk_items.size();
    dp.n_combine = (int32_t)pl.combine.size();
    dp.n_parts = pl.n_parts;
    dp.num_blocks = p->cfg.num_blocks;
    dp.decode_grid = pl.decode_grid;
    dp.decode_packed = pl.decode_packed;
    dp.chunk_single = pl.chunk_single;
  } else if (st != p->upload_stream) {
    cudaError_t e = cudaStreamWaitEvent(st, p->upload_ev, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
  }
  p->use_stream(st);
  return RBKV_OK;
}

rbkv_status check_config(const rbkv_config* c) {
  if (!c) return fail(RBKV_ERR_INVALID, "config is NULL");
  if (c->num_heads_q < 1 || c->num_heads_kv < 1 || c->num_heads_q % c->num_heads_kv)
    return fail(RBKV_ERR_INVALID, "num_heads_q must be a positive multiple of num_heads_kv");
  if (c->block_size < 1 || c->num_blocks < 0)
    return fail(RBKV_ERR_INVALID, "block_size must be >= 1 and num_blocks >= 0");
  if ((int64_t)c->num_blocks * c->block_size >= (int64_t)1 << 31)
    return fail(RBKV_ERR_INVALID, "num_blocks * block_size must fit in int32");
  if (c->dtype != RBKV_BF16 && c->dtype != RBKV_F32)
    return fail(RBKV_ERR_INVALID, "dtype must be RBKV_BF16 or RBKV_F32");
  if (c->head_dim < 32 || c->head_dim > 256 || c->head_dim % 32)
    return fail(RBKV_ERR_UNSUPPORTED, "head_dim must be a multiple of 32 in [32, 256]");
  if (c->num_heads_q / c->num_heads_kv > 64)
    return fail(RBKV_ERR_UNSUPPORTED, "at most 64 query heads per KV head");
  return RBKV_OK;
}

}  // namespace

// ---- attention on a pass already on the device, with a given scratch ---------
// Used by the entry point that allocates nothing (rbkv_noalloc.cu): unlike
// rbkv_ragged_attention it never uploads metadata (that would allocate), so
// the pass must already have been on the device (its rbkv_kv_append call).
namespace rbkv {

rbkv_status set_error(rbkv_status st, const char* msg) { return fail(st, msg); }

void note_launches(int64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

rbkv_status attention_on_device(rbkv_pass* p, const void* q, const void* k_cache,
                                const void* v_cache, void* o, void* scratch,
                                size_t scratch_bytes, cudaStream_t st) {
  if (!p) return fail(RBKV_ERR_INVALID, "pass is NULL");
  if (p->slot.empty()) return RBKV_OK;
  if (!q || !k_cache || !v_cache || !o) return fail(RBKV_ERR_INVALID, "NULL tensor");
  if (!p->dev)
    return fail(RBKV_ERR_INVALID,
                "the pass is not on the device yet: call rbkv_kv_append for it first "
                "(this entry point allocates nothing, so it cannot upload metadata)");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != p->device) return fail(RBKV_ERR_INVALID, "pass is bound to another device");
  const size_t need = workspace_bytes_of(*p);
  if (need > scratch_bytes)
    return fail(RBKV_ERR_WORKSPACE, "this pass needs " + std::to_string(need) +
                                        " bytes of scratch; the static scratch holds " +
                                        std::to_string(scratch_bytes));
  if (st != p->upload_stream) {
    e = cudaStreamWaitEvent(st, p->upload_ev, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
  }
  p->use_stream(st);
  const ShapeInfo s = shape_of(p->cfg);
  float* part_o = (float*)scratch;
  float* part_lse = (float*)((char*)scratch + partial_o_bytes(p->plan.n_parts, s));
  const DevPass& dp = p->dp;
  e = cudaSuccess;
  int launched = 0;
  if (dp.n_decode) {
    e = launch_decode_fast(dp, s, q, k_cache, v_cache, o, part_o, part_lse, st, false, true);
    ++launched;
  }
  if (e == cudaSuccess && dp.n_chunk) {
    e = launch_chunk_fast(dp, s, q, k_cache, v_cache, o, part_o, part_lse, st, dp.n_decode > 0,
                          dp.n_decode == 0);
    ++launched;
  }
  if (e == cudaSuccess && dp.n_generic) {
    e = launch_generic_attention(dp, s, q, k_cache, v_cache, o, part_o, part_lse, st);
    ++launched;
  }
  if (e == cudaSuccess && dp.n_combine) {
    e = launch_combine(dp, s, part_o, part_lse, o, st);
    ++launched;
  }
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  g_launches.fetch_add(launched, std::memory_order_relaxed);
  return RBKV_OK;
}

}  // namespace rbkv

// ============================================================================
// C ABI
// ============================================================================
extern "C" {

int32_t rbkv_abi_version(void) { return RBKV_ABI_VERSION; }

const char* rbkv_last_error(void) { return g_err.c_str(); }

rbkv_status rbkv_composer_create(const rbkv_config* cfg, rbkv_composer** out) {
  if (!out) return fail(RBKV_ERR_INVALID, "out is NULL");
  rbkv_status st = check_config(cfg);
  if (st != RBKV_OK) return st;
  try {
    *out = new rbkv_composer(*cfg);
  } catch (...) {
    return fail(RBKV_ERR_INVALID, "out of host memory");
  }
  return RBKV_OK;
}

void rbkv_composer_destroy(rbkv_composer* c) { delete c; }

int32_t rbkv_composer_free_blocks(const rbkv_composer* c) { return c ? c->pool.free_count() : 0; }

rbkv_status rbkv_compose_pass(rbkv_composer* c, int32_t token_budget, int32_t max_chunk,
                              const rbkv_seq_state* states, int32_t n_states, rbkv_pass** out) {
  return rbkv_compose_pass_policy(c, token_budget, max_chunk, RBKV_CHUNK_GREEDY, states,
                                  n_states, out);
}

rbkv_status rbkv_compose_pass_policy(rbkv_composer* c, int32_t token_budget, int32_t max_chunk,
                                     int32_t chunk_policy, const rbkv_seq_state* states,
                                     int32_t n_states, rbkv_pass** out) {
  rbkv::NvtxRange nvtx_range("rbkv_compose_pass");
  if (!c || !out) return fail(RBKV_ERR_INVALID, "composer or out is NULL");
  if (chunk_policy != RBKV_CHUNK_GREEDY && chunk_policy != RBKV_CHUNK_EQUAL)
    return fail(RBKV_ERR_INVALID, "unknown chunk policy");
  if (token_budget < 0) return fail(RBKV_ERR_INVALID, "token budget must be >= 0");
  if (n_states < 0 || (n_states > 0 && !states))
    return fail(RBKV_ERR_INVALID, "states must hold n_states entries");
  try {
    std::unordered_set<int64_t> ids;
    ids.reserve((size_t)n_states * 2);
    for (int32_t i = 0; i < n_states; ++i) {
      const rbkv_seq_state& q = states[i];
      if (!ids.insert(q.seq_id).second)
        return fail(RBKV_ERR_INVALID, "sequence " + std::to_string(q.seq_id) + " listed twice");
      if (q.prompt_len < 1 || q.prompt_len > kMaxTokens || q.seen < 0 || q.seen > kMaxTokens)
        return fail(RBKV_ERR_INVALID, "sequence " + std::to_string(q.seq_id) +
                                          ": prompt_len must be in [1, 2^30] and seen in [0, 2^30]");
      auto it = c->tokens.find(q.seq_id);
      int32_t have = it == c->tokens.end() ? 0 : it->second;
      if (q.seen != have)
        return fail(RBKV_ERR_INVALID, "sequence " + std::to_string(q.seq_id) + ": seen=" +
                                          std::to_string(q.seen) + " but the cache holds " +
                                          std::to_string(have) + " tokens");
    }
    // generation tokens first, then prompt chunks; both in list order
    std::vector<int32_t> take((size_t)n_states, 0);
    int32_t left = token_budget;
    for (int32_t i = 0; i < n_states && left > 0; ++i)
      if (states[i].seen >= states[i].prompt_len) { take[i] = 1; --left; }
    for (int32_t i = 0; i < n_states; ++i) {
      const rbkv_seq_state& q = states[i];
      if (q.seen >= q.prompt_len) continue;
      const int32_t rem = q.prompt_len - q.seen;
      int32_t allow = left;
      if (max_chunk > 0 && allow > max_chunk) allow = max_chunk;
      int32_t n = rem < allow ? rem : allow;
      if (chunk_policy == RBKV_CHUNK_EQUAL && allow > 0 && rem > allow) {
        // the fewest chunks of at most `allow` tokens, all of (near-)equal size
        const int32_t k = ceil_div(rem, allow);
        n = ceil_div(rem, k);
      }
      take[i] = n;
      left -= n;
    }
    // blocks: all or nothing
    const int32_t B = c->cfg.block_size;
    int64_t need_total = 0;
    std::vector<int32_t> need((size_t)n_states, 0);
    for (int32_t i = 0; i < n_states; ++i) {
      if (!take[i]) continue;
      auto it = c->held.find(states[i].seq_id);
      int32_t have = it == c->held.end() ? 0 : (int32_t)it->second.size();
      need[i] = std::max(0, ceil_div((int64_t)states[i].seen + take[i], B) - have);
      need_total += need[i];
    }
    if (need_total > c->pool.free_count())
      return fail(RBKV_ERR_NO_BLOCKS, "pass needs " + std::to_string(need_total) +
                                          " new blocks, " + std::to_string(c->pool.free_count()) +
                                          " free");
    std::unique_ptr<rbkv_pass> p(new rbkv_pass());
    p->cfg = c->cfg;
    p->pinned = c->pinned;
    for (int32_t i = 0; i < n_states; ++i) {
      if (!take[i]) continue;
      const rbkv_seq_state& q = states[i];
      std::vector<int32_t>& blocks = c->held[q.seq_id];
      for (int32_t k = 0; k < need[i]; ++k) blocks.push_back(c->pool.take_lowest());
      const int32_t n = take[i], seen = q.seen, ctx = seen + n;
      c->tokens[q.seq_id] = ctx;
      p->seq_ids.push_back(q.seq_id);
      p->n_new.push_back(n);
      p->seen.push_back(seen);
      p->ctx.push_back(ctx);
      p->q_start.push_back(p->q_start.back() + n);
      const int32_t nb = ceil_div(ctx, B);
      p->block_ids.insert(p->block_ids.end(), blocks.begin(), blocks.begin() + nb);
      p->block_start.push_back(p->block_start.back() + nb);
      for (int32_t pos = seen; pos < ctx; ++pos)
        p->slot.push_back(blocks[pos / B] * B + pos % B);
    }
    *out = p.release();
  } catch (...) {
    return fail(RBKV_ERR_INVALID, "out of host memory");
  }
  return RBKV_OK;
}

double rbkv_latency_at(const int32_t* tokens, const double* latency, int32_t n, int32_t t) {
  // piecewise-linear interpolation of a measured (tokens, latency) profile
  int32_t i = 0;
  while (i + 2 < n && t > tokens[i + 1]) ++i;
  const double f = (double)(t - tokens[i]) / (double)(tokens[i + 1] - tokens[i]);
  return latency[i] + (latency[i + 1] - latency[i]) * f;
}

int32_t rbkv_budget_for_latency(const int32_t* tokens, const double* latency, int32_t n,
                                double bound) {
  if (!tokens || !latency || n < 2) return -1;
  for (int32_t i = 0; i + 1 < n; ++i)
    if (tokens[i + 1] <= tokens[i] || tokens[i] < 0) return -1;
  for (int32_t t = tokens[n - 1]; t >= tokens[0]; --t)
    if (rbkv_latency_at(tokens, latency, n, t) <= bound) return t;
  return 0;
}

rbkv_status rbkv_release_seq(rbkv_composer* c, int64_t seq_id) {
  if (!c) return fail(RBKV_ERR_INVALID, "composer is NULL");
  auto th = c->tokens.find(seq_id);
  auto hb = c->held.find(seq_id);
  if (th == c->tokens.end() && hb == c->held.end())
    return fail(RBKV_ERR_INVALID, "unknown sequence " + std::to_string(seq_id));
  if (hb != c->held.end()) {
    for (int32_t b : hb->second) c->pool.give_back(b);
    c->held.erase(hb);
  }
  if (th != c->tokens.end()) c->tokens.erase(th);
  return RBKV_OK;
}

rbkv_status rbkv_pass_rollback(rbkv_composer* c, const rbkv_pass* p) {
  if (!c || !p) return fail(RBKV_ERR_INVALID, "composer or pass is NULL");
  const size_t S = p->seq_ids.size();
  // all-or-nothing: every sequence must still be exactly where this pass left it
  for (size_t i = 0; i < S; ++i) {
    auto it = c->tokens.find(p->seq_ids[i]);
    if (it == c->tokens.end() || it->second != p->ctx[i])
      return fail(RBKV_ERR_INVALID, "sequence " + std::to_string(p->seq_ids[i]) +
                                        " changed after this pass; roll back later passes first");
  }
  const int32_t B = c->cfg.block_size;
  for (size_t i = S; i-- > 0;) {
    const int64_t sid = p->seq_ids[i];
    std::vector<int32_t>& held = c->held[sid];
    const size_t keep = (size_t)ceil_div(p->seen[i], B);
    while (held.size() > keep) {
      c->pool.give_back(held.back());
      held.pop_back();
    }
    if (p->seen[i] == 0) {
      c->tokens.erase(sid);
      c->held.erase(sid);
    } else {
      c->tokens[sid] = p->seen[i];
    }
  }
  return RBKV_OK;
}

rbkv_status rbkv_pass_get_meta(const rbkv_pass* p, rbkv_pass_meta* v) {
  if (!p || !v) return fail(RBKV_ERR_INVALID, "pass or view is NULL");
  v->num_seqs = (int32_t)p->seq_ids.size();
  v->num_tokens = (int32_t)p->slot.size();
  v->num_block_ids = (int32_t)p->block_ids.size();
  v->block_size = p->cfg.block_size;
  v->seq_ids = p->seq_ids.data();
  v->q_start = p->q_start.data();
  v->n_new = p->n_new.data();
  v->seen = p->seen.data();
  v->ctx = p->ctx.data();
  v->block_start = p->block_start.data();
  v->block_ids = p->block_ids.data();
  v->slot = p->slot.data();
  return RBKV_OK;
}

rbkv_status rbkv_pass_set_split_keys(rbkv_pass* p, int32_t keys) {
  if (!p) return fail(RBKV_ERR_INVALID, "pass is NULL");
  if (keys < 0 || keys % 16) return fail(RBKV_ERR_INVALID, "keys per split must be a multiple of 16");
  if (p->planned) return fail(RBKV_ERR_INVALID, "the pass was already planned by a device call");
  p->split_keys = keys;
  return RBKV_OK;
}

rbkv_status rbkv_pass_set_chunk_items(rbkv_pass* p, int32_t mode) {
  if (!p) return fail(RBKV_ERR_INVALID, "pass is NULL");
  if (mode < RBKV_CHUNK_ITEMS_AUTO || mode > RBKV_CHUNK_ITEMS_SINGLE)
    return fail(RBKV_ERR_INVALID, "unknown chunk item mode");
  if (p->planned) return fail(RBKV_ERR_INVALID, "the pass was already planned by a device call");
  p->chunk_items = mode;
  return RBKV_OK;
}

rbkv_status rbkv_pass_get_plan(rbkv_pass* p, rbkv_plan_info* info) {
  if (!p || !info) return fail(RBKV_ERR_INVALID, "pass or info is NULL");
  rbkv_status st = ensure_plan(p);
  if (st != RBKV_OK) return st;
  *info = p->plan.info;
  return RBKV_OK;
}

rbkv_status rbkv_pass_plan_for_sms(const rbkv_pass* p, int32_t num_sms, rbkv_plan_info* info) {
  if (!p || !info || num_sms < 1) return fail(RBKV_ERR_INVALID, "bad arguments");
  *info = make_plan(*p, num_sms).info;
  return RBKV_OK;
}

rbkv_status rbkv_debug_corrupt_pass(rbkv_pass* p, int32_t which, int32_t index, int32_t value) {
  if (!p) return fail(RBKV_ERR_INVALID, "pass is NULL");
  if (p->dev || p->planned) return fail(RBKV_ERR_INVALID, "the pass is already on the device");
  std::vector<int32_t>* v = which == 0 ? &p->block_ids : which == 1 ? &p->slot : nullptr;
  if (!v) return fail(RBKV_ERR_INVALID, "which must be 0 (block ids) or 1 (slots)");
  if (index < 0 || (size_t)index >= v->size()) return fail(RBKV_ERR_INVALID, "index out of range");
  (*v)[index] = value;
  return RBKV_OK;
}

rbkv_status rbkv_debug_wait_timeout(rbkv_pass* p, int64_t limit_cycles, rbkv_stream stream) {
  if (!p) return fail(RBKV_ERR_INVALID, "pass is NULL");
  if (!p->dev) return fail(RBKV_ERR_INVALID, "the pass is not on the device");
  if (limit_cycles < 0 || limit_cycles > ((int64_t)1 << 32))
    return fail(RBKV_ERR_INVALID, "limit_cycles must be in [0, 2^32]");
  cudaStream_t st = (cudaStream_t)stream;
  if (st != p->upload_stream) {
    cudaError_t e = cudaStreamWaitEvent(st, p->upload_ev, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");
  }
  p->use_stream(st);
  cudaError_t e = launch_wait_timeout((int32_t*)p->dev, (long long)limit_cycles, st);
  if (e != cudaSuccess) return cuda_fail(e, "wait-timeout launch");
  return RBKV_OK;
}

void rbkv_pass_destroy(rbkv_pass* p) {
  if (!p) return;
  if (p->dev) {
    // the metadata is freed in order after the pass's work on every stream it
    // was used on: the freeing stream first waits for each of the others
    cudaStream_t fs = p->last_stream;
    if (p->streams.size() > 1) {
      cudaEvent_t ev = nullptr;
      if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) == cudaSuccess) {
        for (cudaStream_t st : p->streams) {
          if (st == fs) continue;
          if (cudaEventRecord(ev, st) == cudaSuccess) cudaStreamWaitEvent(fs, ev, 0);
        }
        cudaEventDestroy(ev);
      }
    }
    cudaFreeAsync(p->dev, fs);
  }
  if (p->upload_ev) cudaEventDestroy(p->upload_ev);
  delete p;
}

rbkv_status rbkv_kv_append(rbkv_pass* p, const void* k_new, const void* v_new, void* k_cache,
                           void* v_cache, rbkv_stream stream) {
  rbkv::NvtxRange nvtx_range("rbkv_kv_append");
  if (!p) return fail(RBKV_ERR_INVALID, "pass is NULL");
  if (p->slot.empty()) return RBKV_OK;
  if (!k_new || !v_new || !k_cache || !v_cache) return fail(RBKV_ERR_INVALID, "NULL tensor");
  cudaStream_t st = (cudaStream_t)stream;
  rbkv_status rs = ensure_device(p, st);
  if (rs != RBKV_OK) return rs;
  const ShapeInfo s = shape_of(p->cfg);
  cudaError_t e = launch_counted(RBKV_KERNEL_KV_APPEND, st, [&] {
    return launch_kv_append(p->dp, s, k_new, v_new, k_cache, v_cache, st, !g_prof.on);
  });
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  return RBKV_OK;
}

size_t rbkv_attention_workspace_bytes(rbkv_pass* p) {
  if (!p || ensure_plan(p) != RBKV_OK) return 0;
  return workspace_bytes_of(*p);
}

rbkv_status rbkv_ragged_attention(rbkv_pass* p, const void* q, const void* k_cache,
                                  const void* v_cache, void* o, void* workspace,
                                  size_t workspace_bytes, rbkv_stream stream) {
  rbkv::NvtxRange nvtx_range("rbkv_ragged_attention");
  if (!p) return fail(RBKV_ERR_INVALID, "pass is NULL");
  if (p->slot.empty()) return RBKV_OK;
  if (!q || !k_cache || !v_cache || !o) return fail(RBKV_ERR_INVALID, "NULL tensor");
  rbkv_status rs = ensure_plan(p);
  if (rs != RBKV_OK) return rs;
  const size_t need = workspace_bytes_of(*p);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(RBKV_ERR_WORKSPACE, "workspace needs " + std::to_string(need) + " bytes");
  if (need > 0 && ((uintptr_t)workspace % 256))
    return fail(RBKV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  rs = ensure_device(p, st);
  if (rs != RBKV_OK) return rs;
  const ShapeInfo s = shape_of(p->cfg);
  float* part_o = (float*)workspace;
  float* part_lse = need ? (float*)((char*)workspace + partial_o_bytes(p->plan.n_parts, s)) : nullptr;
  const DevPass& dp = p->dp;
  cudaError_t e = cudaSuccess;
  // Kernels overlap their predecessor in the stream through programmatic
  // dependent launch (not while per-launch events are recorded).  Each waits
  // for its predecessor before touching memory it might share with it: the
  // decode kernel before any global access; the chunk kernel too, unless its
  // predecessor is this call's decode kernel (which lets it start only once
  // everything before the decode kernel has finished).  The decode grid goes
  // first and fills every SM; chunk tiles take SMs as decode CTAs finish.
  const bool overlap = !g_prof.on;
  if (dp.n_decode)
    e = launch_counted(RBKV_KERNEL_DECODE, st, [&] {
      return launch_decode_fast(dp, s, q, k_cache, v_cache, o, part_o, part_lse, st, overlap,
                                true);
    });
  if (e == cudaSuccess && dp.n_chunk)
    e = launch_counted(RBKV_KERNEL_CHUNK, st, [&] {
      return launch_chunk_fast(dp, s, q, k_cache, v_cache, o, part_o, part_lse, st, overlap,
                               dp.n_decode == 0);
    });
  if (e == cudaSuccess && dp.n_generic)
    e = launch_counted(RBKV_KERNEL_GENERIC, st, [&] {
      return launch_generic_attention(dp, s, q, k_cache, v_cache, o, part_o, part_lse, st);
    });
  if (e == cudaSuccess && dp.n_combine)
    e = launch_counted(RBKV_KERNEL_COMBINE, st,
                       [&] { return launch_combine(dp, s, part_o, part_lse, o, st); });
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return RBKV_OK;
}

}  // extern "C"

namespace {

// Wait for `st`, then read and clear the four device status words at `dev`.
rbkv_status read_device_status(void* dev, cudaStream_t st) {
  int32_t words[4] = {0, 0, 0, 0};
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemcpy(words, dev, sizeof(words), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(dev, 0, sizeof(words));
  if (e != cudaSuccess) return cuda_fail(e, "device status read");
  const int32_t word = words[0];
  if (word == kDevBounds) return fail(RBKV_ERR_DEVICE_BOUNDS, "a kernel met an out-of-range block id");
  if (word == kDevTimeout)
    return fail(RBKV_ERR_TIMEOUT, "a bounded device wait gave up (site " + std::to_string(words[1]) +
                                      ", index " + std::to_string(words[2]) + ", block " +
                                      std::to_string(words[3] & 0xFFFF) + "," +
                                      std::to_string(words[3] >> 16) + ")");
  if (word != 0) return fail(RBKV_ERR_CUDA, "unknown device status " + std::to_string(word));
  return RBKV_OK;
}

}  // namespace

extern "C" {

rbkv_status rbkv_pass_device_status(rbkv_pass* p, rbkv_stream stream) {
  if (!p) return fail(RBKV_ERR_INVALID, "pass is NULL");
  if (!p->dev) return RBKV_OK;
  return read_device_status(p->dev, (cudaStream_t)stream);
}

// ---------------------------------------------------------------------------
// frames
// ---------------------------------------------------------------------------
}  // extern "C"

struct rbkv_frame {
  rbkv_config cfg{};
  rbkv_frame_caps caps{};
  int device = -1;
  int sms = 0;
  int32_t* dev = nullptr;   // device words: status[4] | counts[8] | sections
  size_t words = 0;
  size_t o_slot = 0, o_blocks = 0, o_dec = 0, o_chunk = 0, o_items = 0, o_comb = 0;
  int32_t max_items = 0;   // chunk work items: max_chunk_tiles x num_heads_q
  static constexpr int kStages = 4;
  int32_t* host[kStages] = {};   // pinned staging, same layout
  cudaEvent_t ev[kStages] = {};
  int next = 0;
  DevPass dp{};
  ~rbkv_frame() {
    for (int i = 0; i < kStages; ++i) {
      if (ev[i]) { cudaEventSynchronize(ev[i]); cudaEventDestroy(ev[i]); }
      if (host[i]) cudaFreeHost(host[i]);
    }
    if (dev) cudaFree(dev);
  }
};

namespace {

bool same_config(const rbkv_config& a, const rbkv_config& b) {
  return a.num_heads_q == b.num_heads_q && a.num_heads_kv == b.num_heads_kv &&
         a.head_dim == b.head_dim && a.block_size == b.block_size && a.dtype == b.dtype &&
         a.num_blocks == b.num_blocks;
}

size_t align4(size_t w) { return (w + 3) / 4 * 4; }

}  // namespace

extern "C" {

rbkv_status rbkv_frame_create(const rbkv_config* cfg, const rbkv_frame_caps* caps,
                              rbkv_frame** out, rbkv_frame_caps* caps_out) {
  if (!out || !caps) return fail(RBKV_ERR_INVALID, "caps or out is NULL");
  *out = nullptr;
  rbkv_status rs = check_config(cfg);
  if (rs != RBKV_OK) return rs;
  const ShapeInfo s = shape_of(*cfg);
  if (cfg->dtype != RBKV_BF16 || !decode_fast_supported(s) || !chunk_fast_supported(s))
    return fail(RBKV_ERR_UNSUPPORTED, "frames need a shape served by the tensor-core kernels");
  rbkv_frame_caps c = *caps;
  if (c.max_tokens < 1) return fail(RBKV_ERR_INVALID, "max_tokens must be >= 1");
  if (c.max_seqs < 0 || c.max_blocks < 0 || c.max_decode_items < 0 || c.max_chunk_tiles < 0 ||
      c.max_combine_rows < 0 || c.max_parts < 0 || c.packed_units < 0 || c.packed_units > 1 ||
      c.chunk_items < RBKV_CHUNK_ITEMS_AUTO || c.chunk_items > RBKV_CHUNK_ITEMS_SINGLE)
    return fail(RBKV_ERR_INVALID, "capacities must be >= 0");
  int dev = -1, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "device query");
  const int64_t slots = (int64_t)sms * decode_ctas_per_sm(s);
  auto clamp = [](int64_t v) { return (int32_t)std::min<int64_t>(v, 1 << 28); };
  if (!c.max_seqs) c.max_seqs = c.max_tokens;
  if (!c.max_blocks) c.max_blocks = std::max(1, cfg->num_blocks);
  if (!c.max_decode_items)
    c.max_decode_items = clamp(4 * slots + (int64_t)c.max_seqs * s.H_kv);
  if (!c.max_chunk_tiles)   // the chunk grid is persistent: capacity costs nothing at launch
    c.max_chunk_tiles = clamp(std::max<int64_t>((int64_t)ceil_div(c.max_tokens, kChunkTileRows) +
                                                    c.max_seqs,
                                                ceil_div(sms, s.H_q)));
  if (!c.max_combine_rows) c.max_combine_rows = clamp((int64_t)c.max_tokens * s.H_kv);
  if (c.chunk_items == RBKV_CHUNK_ITEMS_AUTO) {
    // the grouping the planner would take for a pass of max_tokens prompt rows
    const int64_t tiles = ceil_div(c.max_tokens, kChunkTileRows);
    const int64_t pairs =
        s.g >= 2 ? tiles * s.H_kv * ceil_div(s.g, 2) : ceil_div(tiles, 2) * s.H_q;
    c.chunk_items = pairs >= sms ? RBKV_CHUNK_ITEMS_PAIRS : RBKV_CHUNK_ITEMS_SINGLE;
  }
  if (!c.max_parts)
    c.max_parts = clamp((int64_t)c.max_decode_items +
                        (int64_t)c.max_tokens * s.H_kv * std::max(1, sms / s.H_q));
  std::unique_ptr<rbkv_frame> f(new rbkv_frame);
  f->cfg = *cfg;
  f->caps = c;
  f->device = dev;
  f->sms = sms;
  size_t w = 12;  // status words, counts
  f->o_slot = w;   w = align4(w + (size_t)c.max_tokens);
  f->o_blocks = w; w = align4(w + (size_t)c.max_blocks);
  f->o_dec = w;    w = align4(w + (size_t)c.max_decode_items * (sizeof(WorkItem) / 4));
  f->o_chunk = w;  w = align4(w + (size_t)c.max_chunk_tiles * (sizeof(ChunkTile) / 4));
  f->max_items = (int32_t)std::min<int64_t>((int64_t)c.max_chunk_tiles * s.H_q, 1 << 28);
  f->o_items = w;  w = align4(w + (size_t)f->max_items * (sizeof(ChunkItem) / 4));
  f->o_comb = w;   w = align4(w + (size_t)c.max_combine_rows * (sizeof(CombineRow) / 4));
  f->words = w;
  e = cudaMalloc((void**)&f->dev, w * 4);
  if (e == cudaSuccess) e = cudaMemset(f->dev, 0, w * 4);
  for (int i = 0; e == cudaSuccess && i < rbkv_frame::kStages; ++i) {
    e = cudaHostAlloc((void**)&f->host[i], w * 4, cudaHostAllocDefault);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&f->ev[i], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) return cuda_fail(e, "frame allocation");
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "frame allocation");
  DevPass& dp = f->dp;
  int32_t* base = f->dev;
  dp.status = base;
  dp.counts = base + 4;
  dp.slot = base + f->o_slot;
  dp.block_ids = base + f->o_blocks;
  dp.decode_items = (const WorkItem*)(base + f->o_dec);
  dp.generic_items = nullptr;
  dp.chunk_tiles = (const ChunkTile*)(base + f->o_chunk);
  dp.chunk_items = (const ChunkItem*)(base + f->o_items);
  dp.combine_rows = (const CombineRow*)(base + f->o_comb);
  dp.num_tokens = c.max_tokens;
  dp.n_decode = c.max_decode_items;
  dp.n_generic = 0;
  dp.n_chunk = f->max_items;
  dp.n_combine = c.max_combine_rows;
  dp.n_parts = c.max_parts;
  dp.num_blocks = cfg->num_blocks;
  dp.decode_grid = (int32_t)std::min<int64_t>(slots, c.max_decode_items);
  dp.decode_packed = c.packed_units ? 1 : 0;
  dp.chunk_single = c.chunk_items == RBKV_CHUNK_ITEMS_SINGLE ? 1 : 0;
  if (caps_out) *caps_out = c;
  *out = f.release();
  return RBKV_OK;
}

void rbkv_frame_destroy(rbkv_frame* f) { delete f; }

rbkv_status rbkv_frame_load(rbkv_frame* f, rbkv_pass* p, rbkv_stream stream) {
  rbkv::NvtxRange nvtx_range("rbkv_frame_load");
  if (!f || !p) return fail(RBKV_ERR_INVALID, "frame or pass is NULL");
  if (!same_config(f->cfg, p->cfg)) return fail(RBKV_ERR_INVALID, "pass and frame configs differ");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != f->device) return fail(RBKV_ERR_INVALID, "frame belongs to another device");
  const rbkv_frame_caps& c = f->caps;
  int32_t counts[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const Plan* pl = nullptr;
  if (!p->slot.empty()) {
    if (!p->planned) p->chunk_items = c.chunk_items;   // the frame's grouping
    rbkv_status rs = ensure_plan(p);
    if (rs != RBKV_OK) return rs;
    pl = &p->plan;
    if (pl->chunk_single != f->dp.chunk_single)
      return fail(RBKV_ERR_UNSUPPORTED,
                  "the pass was planned with another grouping of its chunk tiles than the "
                  "frame's");
    auto over = [](const char* what, size_t n, int32_t cap) {
      return fail(RBKV_ERR_WORKSPACE, std::string("pass exceeds the frame's ") + what + " (" +
                                          std::to_string(n) + " > " + std::to_string(cap) + ")");
    };
    if (p->slot.size() > (size_t)c.max_tokens) return over("max_tokens", p->slot.size(), c.max_tokens);
    if (p->seq_ids.size() > (size_t)c.max_seqs) return over("max_seqs", p->seq_ids.size(), c.max_seqs);
    if (p->block_ids.size() > (size_t)c.max_blocks)
      return over("max_blocks", p->block_ids.size(), c.max_blocks);
    if (pl->decode.size() > (size_t)c.max_decode_items)
      return over("max_decode_items", pl->decode.size(), c.max_decode_items);
    if (pl->chunk.size() > (size_t)c.max_chunk_tiles)
      return over("max_chunk_tiles", pl->chunk.size(), c.max_chunk_tiles);
    if (pl->chunk_items.size() > (size_t)f->max_items)
      return over("chunk items (max_chunk_tiles x num_heads_q)", pl->chunk_items.size(),
                  f->max_items);
    if (pl->combine.size() > (size_t)c.max_combine_rows)
      return over("max_combine_rows", pl->combine.size(), c.max_combine_rows);
    if (pl->n_parts > c.max_parts) return over("max_parts", (size_t)pl->n_parts, c.max_parts);
    if (!pl->generic.empty()) return fail(RBKV_ERR_UNSUPPORTED, "pass has CUDA-core work items");
    if (pl->decode_packed && !c.packed_units)
      return fail(RBKV_ERR_UNSUPPORTED,
                  "pass has short prompt chunks packed into decode units; the frame was "
                  "created without packed_units");
    counts[kCountTokens] = (int32_t)p->slot.size();
    counts[kCountDecode] = (int32_t)pl->decode.size();
    counts[kCountChunk] = (int32_t)pl->chunk_items.size();
    counts[kCountCombine] = (int32_t)pl->combine.size();
  }
  const int k = f->next;
  f->next = (f->next + 1) % rbkv_frame::kStages;
  e = cudaEventSynchronize(f->ev[k]);  // the last copy out of this staging buffer
  if (e != cudaSuccess) return cuda_fail(e, "frame staging");
  int32_t* h = f->host[k];
  cudaStream_t st = (cudaStream_t)stream;
  std::memcpy(h + 4, counts, sizeof(counts));
  size_t head_end = 12;
  if (pl) {
    std::memcpy(h + f->o_slot, p->slot.data(), p->slot.size() * 4);
    std::memcpy(h + f->o_blocks, p->block_ids.data(), p->block_ids.size() * 4);
    head_end = f->o_blocks + p->block_ids.size();
  }
  // counts, slots and block tables in one copy (not the status words), then
  // the used part of each work list
  e = cudaMemcpyAsync(f->dev + 4, h + 4, (head_end - 4) * 4, cudaMemcpyHostToDevice, st);
  auto section = [&](size_t off, const void* src, size_t bytes) {
    if (e != cudaSuccess || bytes == 0) return;
    std::memcpy(h + off, src, bytes);
    e = cudaMemcpyAsync(f->dev + off, h + off, bytes, cudaMemcpyHostToDevice, st);
  };
  if (pl) {
    section(f->o_dec, pl->decode.data(), pl->decode.size() * sizeof(WorkItem));
    section(f->o_chunk, pl->chunk.data(), pl->chunk.size() * sizeof(ChunkTile));
    section(f->o_items, pl->chunk_items.data(), pl->chunk_items.size() * sizeof(ChunkItem));
    section(f->o_comb, pl->combine.data(), pl->combine.size() * sizeof(CombineRow));
  }
  if (e == cudaSuccess) e = cudaEventRecord(f->ev[k], st);
  if (e != cudaSuccess) return cuda_fail(e, "frame upload");
  return RBKV_OK;
}

rbkv_status rbkv_frame_kv_append(rbkv_frame* f, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, rbkv_stream stream) {
  rbkv::NvtxRange nvtx_range("rbkv_frame_kv_append");
  if (!f) return fail(RBKV_ERR_INVALID, "frame is NULL");
  if (!k_new || !v_new || !k_cache || !v_cache) return fail(RBKV_ERR_INVALID, "NULL tensor");
  cudaStream_t st = (cudaStream_t)stream;
  const ShapeInfo s = shape_of(f->cfg);
  cudaError_t e = launch_counted(RBKV_KERNEL_KV_APPEND, st, [&] {
    return launch_kv_append(f->dp, s, k_new, v_new, k_cache, v_cache, st, !g_prof.on);
  });
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  return RBKV_OK;
}

size_t rbkv_frame_workspace_bytes(const rbkv_frame* f) {
  if (!f) return 0;
  const ShapeInfo s = shape_of(f->cfg);
  return partial_o_bytes(f->caps.max_parts, s) + partial_lse_bytes(f->caps.max_parts, s);
}

rbkv_status rbkv_frame_attention(rbkv_frame* f, const void* q, const void* k_cache,
                                 const void* v_cache, void* o, void* workspace,
                                 size_t workspace_bytes, rbkv_stream stream) {
  rbkv::NvtxRange nvtx_range("rbkv_frame_attention");
  if (!f) return fail(RBKV_ERR_INVALID, "frame is NULL");
  if (!q || !k_cache || !v_cache || !o) return fail(RBKV_ERR_INVALID, "NULL tensor");
  const size_t need = rbkv_frame_workspace_bytes(f);
  if (!workspace || workspace_bytes < need)
    return fail(RBKV_ERR_WORKSPACE, "frame workspace needs " + std::to_string(need) + " bytes");
  if ((uintptr_t)workspace % 256) return fail(RBKV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  const ShapeInfo s = shape_of(f->cfg);
  float* part_o = (float*)workspace;
  float* part_lse = (float*)((char*)workspace + partial_o_bytes(f->caps.max_parts, s));
  const DevPass& dp = f->dp;
  // the same launch sequence as rbkv_ragged_attention with every kernel
  // present: the decode grid always precedes the chunk grid (its CTAs without
  // a unit leave; chunk CTAs without a tile wait for the decode grid and leave)
  const bool overlap = !g_prof.on;
  cudaError_t e = launch_counted(RBKV_KERNEL_DECODE, st, [&] {
    return launch_decode_fast(dp, s, q, k_cache, v_cache, o, part_o, part_lse, st, overlap,
                              true);
  });
  if (e == cudaSuccess)
    e = launch_counted(RBKV_KERNEL_CHUNK, st, [&] {
      return launch_chunk_fast(dp, s, q, k_cache, v_cache, o, part_o, part_lse, st, overlap,
                               false);
    });
  if (e == cudaSuccess)
    e = launch_counted(RBKV_KERNEL_COMBINE, st,
                       [&] { return launch_combine(dp, s, part_o, part_lse, o, st); });
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return RBKV_OK;
}

rbkv_status rbkv_frame_device_status(rbkv_frame* f, rbkv_stream stream) {
  if (!f) return fail(RBKV_ERR_INVALID, "frame is NULL");
  return read_device_status(f->dev, (cudaStream_t)stream);
}

int64_t rbkv_kernel_launches(void) { return g_launches.load(); }

void rbkv_profile_enable(int32_t on) { g_prof.on = on != 0; }

rbkv_status rbkv_profile_read(int32_t kind, double* total_ms, int64_t* launches) {
  if (kind < 0 || kind >= RBKV_KERNEL_KINDS || !total_ms || !launches)
    return fail(RBKV_ERR_INVALID, "bad arguments");
  double t = 0.0;
  for (auto& pr : g_prof.rec[kind]) {
    cudaError_t e = cudaEventSynchronize(pr.second);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, pr.first, pr.second);
    if (e != cudaSuccess) return cuda_fail(e, "profile event");
    t += ms;
  }
  *total_ms = t;
  *launches = (int64_t)g_prof.rec[kind].size();
  return RBKV_OK;
}

void rbkv_profile_reset(void) { g_prof.reset(); }

}  // extern "C"
