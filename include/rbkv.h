/*
 * rbkv.h - C ABI of librbkv: the data-parallel hot path of a Dynamic SplitFuse
 * serving pass on one GB300 (sm_103a).
 *
 * A pass is composed on the host to a fixed token budget, its new K/V rows are
 * appended into a blocked (paged) cache, and ragged causal attention is run
 * for every token of the pass against its sequence's cached keys.
 *
 *   DeepSpeed-FastGen paper summary page, "Summary" and idea I3: every forward
 *     pass holds a fixed token budget; long prompts are cut into chunks over
 *     several passes, and decode tokens and small prompts take the rest.
 *   FastGen guide, "Paged KV Memory Management": the cache is non-contiguous
 *     fixed-size blocks reached through block tables, read directly by the
 *     attention kernels.
 *   FastGen guide, "Dynamic SplitKV Attention": a decode token's keys are split
 *     across SMs by sequence length; each split yields a partial output and a
 *     log-sum-exp, and a small reduction kernel combines them.
 *   FastGen guide, "The Continuous Batching Dilemma": prompt work is a dense
 *     contraction for the tensor cores, decode work is bound by HBM.
 *
 * Conventions for every call:
 *  - Nothing is thrown across this ABI.  Every call returns an rbkv_status;
 *    on error it changes no state and launches nothing, and rbkv_last_error()
 *    returns a message for the calling thread.
 *  - Device pointers are plain CUDA device addresses on the current device,
 *    owned by the caller, contiguous, 16-byte aligned.  Host pointers are
 *    ordinary process memory.  Streams are CUDA stream handles
 *    (cudaStream_t); NULL is the legacy default stream.
 *  - Launches are asynchronous on the given stream.
 *  - A composer and the passes it made are not thread-safe; use one thread per
 *    composer at a time.
 *  - Shapes and element types come from the composer's rbkv_config.  Supported:
 *    RBKV_BF16 or RBKV_F32 elements, head_dim a multiple of 32 up to 256,
 *    num_heads_q a multiple of num_heads_kv (at most 64 query heads per KV
 *    head).
 *
 * Layouts (row-major, innermost last):
 *    Q, O          [T][H_q][D]     element type of the config
 *    K_new, V_new  [T][H_kv][D]
 *    K/V cache     [num_blocks][H_kv][B][D]   (separate K and V arrays)
 *  Token position p of a sequence lives in block table[p / B], slot p % B.
 *  Query head h reads KV head h / (H_q / H_kv).
 */
#ifndef RBKV_H
#define RBKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RBKV_ABI_VERSION 3

typedef enum {
  RBKV_OK = 0,
  RBKV_ERR_INVALID = -1,       /* bad argument, state or sequence id */
  RBKV_ERR_NO_BLOCKS = -2,     /* block pool too small for the pass; nothing changed */
  RBKV_ERR_CUDA = -3,          /* a CUDA runtime/driver call failed (message has it) */
  RBKV_ERR_DEVICE_BOUNDS = -4, /* a kernel met an out-of-range index and skipped it */
  RBKV_ERR_UNSUPPORTED = -5,   /* shape or type outside what the kernels handle */
  RBKV_ERR_WORKSPACE = -6,     /* workspace missing or smaller than required */
  RBKV_ERR_TIMEOUT = -7        /* a bounded device-side wait gave up */
} rbkv_status;

typedef enum { RBKV_BF16 = 0, RBKV_F32 = 1 } rbkv_dtype;

/* Shape of one attention layer and the size of the block pool. */
typedef struct {
  int32_t num_heads_q;
  int32_t num_heads_kv;
  int32_t head_dim;
  int32_t block_size;   /* B, tokens per cache block */
  int32_t dtype;        /* rbkv_dtype of Q, K, V, O and the caches */
  int32_t num_blocks;   /* blocks in the pool (ids 0 .. num_blocks-1) */
} rbkv_config;

/* One request as the caller lists it for a pass.
 * seen < prompt_len : prefilling; the pass may take a chunk of its prompt.
 * seen >= prompt_len: decoding; the pass may take its one generation token.
 * seen must equal the number of tokens the composer has recorded for the id
 * (0 for an id it has not seen). */
typedef struct {
  int64_t seq_id;
  int32_t prompt_len;
  int32_t seen;
} rbkv_seq_state;

typedef struct rbkv_composer rbkv_composer;
typedef struct rbkv_pass rbkv_pass;
typedef struct CUstream_st* rbkv_stream;   /* same type as cudaStream_t */

/* Read-only host view of a pass's ragged-batch metadata.  S = num_seqs
 * scheduled sequences in the caller's list order, T = num_tokens.
 * Valid until rbkv_pass_destroy. */
typedef struct {
  int32_t num_seqs;
  int32_t num_tokens;
  int32_t num_block_ids;
  int32_t block_size;
  const int64_t* seq_ids;     /* [S] */
  const int32_t* q_start;     /* [S+1] first pass row of each sequence; q_start[S] = T */
  const int32_t* n_new;       /* [S] tokens of the sequence in this pass (>= 1) */
  const int32_t* seen;        /* [S] tokens cached before the pass */
  const int32_t* ctx;         /* [S] seen + n_new */
  const int32_t* block_start; /* [S+1] offsets into block_ids */
  const int32_t* block_ids;   /* block table of sequence s: block_ids[block_start[s] ..] */
  const int32_t* slot;        /* [T] block_id * B + offset of each pass row's K/V */
} rbkv_pass_meta;

/* How the attention work of a pass was split (for tests and reports). */
typedef struct {
  int32_t num_sms;            /* SMs of the device the plan was made for */
  int32_t decode_rows;        /* pass rows with one new token (decode path) */
  int32_t decode_items;       /* (row, kv head, key split) work units */
  int32_t max_splits;         /* largest number of splits of one (row, kv head) */
  int32_t split_keys;         /* keys per split used by the plan */
  int32_t partials;           /* partial outputs written to the workspace */
  int32_t chunk_rows;         /* pass rows of multi-token prompt chunks */
  int32_t chunk_tiles;        /* tensor-core query tiles (128 rows, one key piece) */
  int32_t generic_items;      /* work units on the CUDA-core path */
  int32_t fast_decode;        /* 1 if the TMA/tensor-core decode kernel is used */
  int32_t fast_chunk;         /* 1 if the tcgen05 chunk kernel is used */
  int32_t chunk_items;        /* tensor-core work items: one or two query tiles
                                 sharing the K/V tiles they read */
  int32_t chunk_single;       /* 1 if every work item holds one query tile */
  int32_t chunk_steps_total;  /* chunk work in key-tile steps (each item: its
                                 tiles' key tiles, plus one) */
  int32_t chunk_steps_max;    /* the most of it that one CTA of the persistent
                                 chunk grid walks, after the items' placement
                                 was balanced over min(items, SMs) CTAs */
  int32_t decode_grid;        /* CTAs of the persistent decode grid */
  int32_t decode_keys_total;  /* keys the decode-kernel units cover (each unit:
                                 its key range; a KV head's keys count once
                                 per head) */
  int32_t decode_keys_max;    /* the most of them one CTA of the decode grid
                                 walks, after the units' placement */
} rbkv_plan_info;

/* Library ABI version (RBKV_ABI_VERSION). */
int32_t rbkv_abi_version(void);

/* Message of the last failed call on this thread ("" if none). */
const char* rbkv_last_error(void);

/* ---- composition (host only; FastGen paper summary page, Summary) -------- */

/* Create a composer with an empty pool of cfg->num_blocks blocks.
 * Errors: RBKV_ERR_INVALID for a bad config, RBKV_ERR_UNSUPPORTED for shapes
 * the kernels cannot run. */
rbkv_status rbkv_composer_create(const rbkv_config* cfg, rbkv_composer** out);

/* Free a composer.  Passes it made stay valid and must still be destroyed. */
void rbkv_composer_destroy(rbkv_composer* c);

/* Compose one pass from n_states requests in list order.
 * token_budget >= 0: the pass holds min(budget, demand) tokens, demand being
 *   one token per decoding request plus each prefilling request's remaining
 *   prompt (capped at max_chunk when max_chunk > 0).
 * Generation tokens are admitted first, in list order; then each prefilling
 * request takes min(remaining prompt, max_chunk, remaining budget) in list
 * order.  Scheduled sequences are laid out in list order.  Each receives the
 * blocks its new context needs, lowest free block id first.
 * Errors: RBKV_ERR_INVALID (negative budget, duplicate id, prompt_len < 1,
 * seen not matching the recorded context), RBKV_ERR_NO_BLOCKS (pool short; no
 * state changed).  *out receives a new pass (owned by the caller; destroy it
 * with rbkv_pass_destroy), also for an empty pass. */
rbkv_status rbkv_compose_pass(rbkv_composer* c, int32_t token_budget, int32_t max_chunk,
                              const rbkv_seq_state* states, int32_t n_states,
                              rbkv_pass** out);

/* Undo what composing pass p did to the composer: each of its sequences goes
 * back to its `seen` tokens and returns the blocks the pass gave it (a
 * sequence first seen in p is forgotten).  The caller's cache contents are not
 * touched.  Passes must be rolled back newest first; if a sequence of p was
 * changed by a later pass, returns RBKV_ERR_INVALID and changes nothing.
 * Composing the same states again afterwards yields the same metadata. */
rbkv_status rbkv_pass_rollback(rbkv_composer* c, const rbkv_pass* p);

/* Chunk policies for rbkv_compose_pass_policy. */
typedef enum {
  RBKV_CHUNK_GREEDY = 0, /* a prefilling request takes min(remaining prompt, max_chunk,
                            remaining budget): the pass holds exactly the budget when
                            demand allows (rbkv_compose_pass) */
  RBKV_CHUNK_EQUAL = 1   /* a prompt longer than what the pass allows it (a = min(max_chunk,
                            remaining budget)) is cut into the fewest chunks of at most a
                            tokens, all of near-equal size: this pass takes
                            ceil(r / ceil(r / a)) of its r remaining tokens */
} rbkv_chunk_policy;

/* rbkv_compose_pass with a chunk policy.  RBKV_CHUNK_EQUAL follows the FastGen
 * paper summary page, idea I2: throughput is concave in the tokens of a pass,
 * so a pool of prompt tokens is best spread evenly over the passes it needs.
 * The prompt still finishes in the same number of passes as with
 * RBKV_CHUNK_GREEDY; a pass may then hold fewer tokens than the budget.
 * Errors: as rbkv_compose_pass, and RBKV_ERR_INVALID for an unknown policy. */
rbkv_status rbkv_compose_pass_policy(rbkv_composer* c, int32_t token_budget, int32_t max_chunk,
                                     int32_t chunk_policy, const rbkv_seq_state* states,
                                     int32_t n_states, rbkv_pass** out);

/* A latency-bounded token budget (FastGen paper summary page, idea I1: the
 * latency of a forward pass depends mainly on its token count; FastGen guide,
 * "Prompt-Decode Decoupling": keep each iteration under a latency bound).
 * tokens[0..n-1] (strictly increasing, >= 0) and latency[0..n-1] are a measured
 * profile; the predicted latency of t tokens is the linear interpolation
 * between the two profile points around t (rbkv_latency_at).  Returns the
 * largest t in [tokens[0], tokens[n-1]] whose predicted latency is <= bound,
 * 0 if there is none, -1 for a bad profile (n < 2, not increasing, NULL). */
int32_t rbkv_budget_for_latency(const int32_t* tokens, const double* latency, int32_t n,
                                double bound);

/* Predicted latency of t tokens from a profile (as above; t within the profile
 * range, the profile valid). */
double rbkv_latency_at(const int32_t* tokens, const double* latency, int32_t n, int32_t t);

/* Return every block of seq_id to the pool and forget the sequence.
 * Errors: RBKV_ERR_INVALID for an unknown id. */
rbkv_status rbkv_release_seq(rbkv_composer* c, int64_t seq_id);

/* Free blocks in the pool. */
int32_t rbkv_composer_free_blocks(const rbkv_composer* c);

/* Host view of a pass's metadata (pointers owned by the pass). */
rbkv_status rbkv_pass_get_meta(const rbkv_pass* p, rbkv_pass_meta* view);

/* Override the key-split length of the decode plan: keys per split, a positive
 * multiple of 16 (0 = automatic from context lengths and the SM count).  Must
 * be called before the pass's first device call.  Results do not depend on it
 * beyond floating-point rounding. */
rbkv_status rbkv_pass_set_split_keys(rbkv_pass* p, int32_t keys_per_split);

/* How prompt-chunk tiles are grouped into tensor-core work items. */
typedef enum {
  RBKV_CHUNK_ITEMS_AUTO = 0,   /* pairs when there are at least as many as SMs, else one
                                  tile per item */
  RBKV_CHUNK_ITEMS_PAIRS = 1,  /* two tiles that read the same K/V tiles per item (two
                                  query heads of a KV group, or two consecutive row tiles
                                  when the group has one head) */
  RBKV_CHUNK_ITEMS_SINGLE = 2  /* one tile and query head per item */
} rbkv_chunk_items;

/* Override how the pass's prompt-chunk tiles are grouped into work items
 * (rbkv_chunk_items); must be called before the pass's first device call.
 * Results do not depend on it beyond floating-point rounding. */
rbkv_status rbkv_pass_set_chunk_items(rbkv_pass* p, int32_t mode);

/* Plan summary; makes the plan for the current device if not made yet. */
rbkv_status rbkv_pass_get_plan(rbkv_pass* p, rbkv_plan_info* info);

/* Plan summary for a hypothetical device with num_sms SMs (host only; the
 * pass's own plan is not changed).  For inspecting the split planner. */
rbkv_status rbkv_pass_plan_for_sms(const rbkv_pass* p, int32_t num_sms, rbkv_plan_info* info);

/* Free a pass.  Its device metadata is released in stream order after the
 * work launched with it on every stream it was used on (the last of them waits
 * for the others), so all those streams must still exist. */
void rbkv_pass_destroy(rbkv_pass* p);

/* ---- device steps ---------------------------------------------------------- */

/* Append the pass's new K and V rows into the caches (FastGen guide, "Paged KV
 * Memory Management"): for pass row t of sequence s at position p,
 * k_cache[table_s[p/B]][h][p%B][:] = k_new[t][h][:] (same for V), all h.
 * k_new, v_new: [T][H_kv][D]; k_cache, v_cache: [num_blocks][H_kv][B][D].
 * The first device call of a pass uploads its metadata: a small kernel on
 * `stream` copies it from mapped pinned host memory into a stream-ordered
 * device allocation.  A pass is bound to the device current at that call.
 * Errors: RBKV_ERR_INVALID (null pointer with T > 0, other device),
 * RBKV_ERR_CUDA. */
rbkv_status rbkv_kv_append(rbkv_pass* p, const void* k_new, const void* v_new,
                           void* k_cache, void* v_cache, rbkv_stream stream);

/* Bytes of device workspace rbkv_ragged_attention needs for this pass (fp32
 * partial outputs and log-sum-exps of split decode rows); 0 when nothing is
 * split.  Makes the plan for the current device if not made yet. */
size_t rbkv_attention_workspace_bytes(rbkv_pass* p);

/* Ragged causal attention of every pass row (FastGen guide, "Dynamic SplitKV
 * Attention" and Step 3's reference operator; exact softmax attention):
 *   O[t][h][:] = sum_{i<=p} softmax_i(Q[t][h] . K_s[i] / sqrt(D)) V_s[i]
 * for row t of sequence s at position p, keys read through s's block table
 * after this pass's append (call rbkv_kv_append first, same stream).
 * q: [T][H_q][D]; o: [T][H_q][D] (written); caches as above.
 * workspace: device memory of at least rbkv_attention_workspace_bytes(p)
 * bytes (may be NULL when that is 0), 256-byte aligned, owned by the caller;
 * it must not be used by other work until this call's kernels complete.
 * Errors: RBKV_ERR_INVALID, RBKV_ERR_WORKSPACE, RBKV_ERR_CUDA. */
rbkv_status rbkv_ragged_attention(rbkv_pass* p, const void* q, const void* k_cache,
                                  const void* v_cache, void* o, void* workspace,
                                  size_t workspace_bytes, rbkv_stream stream);

/* Ragged attention that allocates nothing.  No counterpart in the paper: this
 * is for callers that cannot call cudaMalloc or any other allocator where they
 * run attention (a fixed device-memory budget handed out up front, a runtime
 * that owns all device memory through its own pool, or a step that must not
 * block or fail on an allocation).  Same computation, inputs and outputs as
 * rbkv_ragged_attention, but the split-KV scratch is a 16 MiB array inside the
 * library (held on every GPU that loads the library until the process exits)
 * instead of a caller workspace.
 *  - The pass must already be on the device: call rbkv_kv_append for it first
 *    (that call uploads its metadata); otherwise RBKV_ERR_INVALID.
 *  - A pass whose scratch need (rbkv_attention_workspace_bytes) exceeds
 *    16 MiB is rejected with RBKV_ERR_WORKSPACE.
 *  - The first call on a device looks up the array's device address for that
 *    device; make that first call before any stream capture.  The address is
 *    kept for the life of the process: after cudaDeviceReset (or anything else
 *    that tears down the device's context) the library's module may load at
 *    another address, so this entry point must not be used on that device
 *    again in the same process.
 *  - All calls share the one array: calls whose kernels overlap on the GPU
 *    race on it.  Order them on one stream (or with events).
 * Calls no cudaMalloc, cudaFree or other allocating routine. */
rbkv_status rbkv_ragged_attention_noalloc(rbkv_pass* p, const void* q, const void* k_cache,
                                          const void* v_cache, void* o, rbkv_stream stream);

/* Wait for `stream`, then read and clear the pass's device status word:
 * RBKV_OK, RBKV_ERR_DEVICE_BOUNDS (a kernel met a block id outside the pool and
 * skipped that access) or RBKV_ERR_TIMEOUT (a bounded wait gave up). */
rbkv_status rbkv_pass_device_status(rbkv_pass* p, rbkv_stream stream);

/* ---- diagnostics: failure detection without a GPU fault ----------------------
 *
 * The kernels never trap: a block id or slot outside the pool is reported in
 * the pass's device status word (RBKV_ERR_DEVICE_BOUNDS) and the access is
 * skipped; every wait on a barrier is bounded and a wait that gives up is
 * reported (RBKV_ERR_TIMEOUT, with the wait site) before the kernel returns.
 * These two calls let tests drive both paths on a real GPU. */

/* Overwrite entry `index` of the pass's block tables (which = 0) or of its
 * slot list (which = 1) with `value`, before the pass's first device call
 * (the composer's own state is not touched; destroy the pass afterwards).
 * Errors: RBKV_ERR_INVALID for a bad which/index, or a pass already on the
 * device. */
rbkv_status rbkv_debug_corrupt_pass(rbkv_pass* p, int32_t which, int32_t index, int32_t value);

/* Launch one CTA on `stream` that waits on a barrier nothing will complete,
 * giving up after `limit_cycles` SM clock cycles (at most 2^32), and reports
 * the timeout (wait site 99) in the pass's status words, as a kernel's own
 * bounded wait would.  The pass must be on the device (after rbkv_kv_append).
 * Read the result with rbkv_pass_device_status. */
rbkv_status rbkv_debug_wait_timeout(rbkv_pass* p, int64_t limit_cycles, rbkv_stream stream);

/* ---- routing over replicas (host only) ------------------------------------
 *
 * InfoQ release note on DeepSpeed-FastGen: throughput scales with the number
 * of replicas behind a load balancer (16 replicas, 23.7 queries/s).  Every
 * replica (one GPU, one composer, one cache) serves its requests on its own;
 * a router only decides which replica takes a request, so there is no
 * exchange between replicas on the data path.  Policy: the replica with the
 * fewest outstanding tokens (prompt tokens not yet prefilled plus output
 * tokens not yet generated, over the requests it holds) takes the next
 * request; ties go to the replica holding fewer requests, then to the lowest
 * index.  Replicas report the tokens each request consumed after every pass
 * (rbkv_router_progress) and its end (rbkv_router_finish).  A router is not
 * thread-safe. */

typedef struct rbkv_router rbkv_router;

/* Errors: RBKV_ERR_INVALID for num_replicas < 1. */
rbkv_status rbkv_router_create(int32_t num_replicas, rbkv_router** out);
void rbkv_router_destroy(rbkv_router* r);

/* Route a new request; *replica receives the replica that takes it.
 * Errors: RBKV_ERR_INVALID (lengths < 1, an id already routed). */
rbkv_status rbkv_router_assign(rbkv_router* r, int64_t request_id, int32_t prompt_len,
                               int32_t output_len, int32_t* replica);

/* `tokens` more of the request's prompt or output were served (at most its
 * outstanding tokens).  Errors: RBKV_ERR_INVALID (unknown id, bad count). */
rbkv_status rbkv_router_progress(rbkv_router* r, int64_t request_id, int32_t tokens);

/* The request ended; its replica's load drops by what it still had
 * outstanding.  Errors: RBKV_ERR_INVALID (unknown id). */
rbkv_status rbkv_router_finish(rbkv_router* r, int64_t request_id);

/* Outstanding tokens / requests held by a replica (-1 for a bad index). */
int64_t rbkv_router_load(const rbkv_router* r, int32_t replica);
int32_t rbkv_router_active(const rbkv_router* r, int32_t replica);

/* ---- frames: one fixed launch sequence for every pass (CUDA graphs) ---------
 *
 * Under Dynamic SplitFuse the passes all have roughly one size (paper
 * summary page, Summary and idea I3; InfoQ release note: passes of a steady
 * size), so a serving loop can record the launches of one pass once, as a
 * CUDA graph, and replay them for every later pass.  A frame makes that
 * possible: it holds a pass's metadata at fixed device addresses, inside
 * capacities fixed when it is created, and its kernel launches are sized by
 * those capacities (the loaded pass's own counts are read on the device).
 * The launches of rbkv_frame_kv_append and rbkv_frame_attention therefore have
 * the same arguments for every pass loaded into the frame; they allocate
 * nothing, wait on no event and never synchronise, so they may be captured.
 * Results are identical to rbkv_kv_append + rbkv_ragged_attention on the same
 * pass (same plan, same kernels).
 *
 * Protocol (all on one stream): rbkv_frame_load(pass) writes the pass's
 * metadata into the frame (host-to-device copies on the stream); then the
 * frame's append and attention launches, directly or replayed from a graph;
 * then the next rbkv_frame_load.  Only bf16 shapes whose decode and chunk rows
 * both take the fast kernels are supported (RBKV_ERR_UNSUPPORTED otherwise). */

typedef struct rbkv_frame rbkv_frame;

/* Capacities of a frame.  0 in any field but max_tokens takes the default:
 *   max_seqs          max_tokens
 *   max_blocks        the pool's num_blocks
 *   max_decode_items  4 x SMs + max_seqs x num_heads_kv (the automatic split
 *                     plan never needs more)
 *   max_chunk_tiles   ceil(max_tokens / 128) + max_seqs, at least ceil(SMs / num_heads_q)
 *   max_combine_rows  max_tokens x num_heads_kv
 *   max_parts         max_decode_items + max_tokens x num_heads_kv x
 *                     max(1, SMs / num_heads_q)
 *   packed_units      0 (passes whose short prompt chunks run as packed decode
 *                     units are refused with RBKV_ERR_UNSUPPORTED)
 *   chunk_items       RBKV_CHUNK_ITEMS_AUTO: pairs when a pass of max_tokens
 *                     prompt rows would give at least as many pairs of tiles
 *                     as SMs, else one tile per item.  Every pass loaded into
 *                     the frame is planned with the frame's grouping (a pass
 *                     already planned with another is refused with
 *                     RBKV_ERR_UNSUPPORTED) and the frame's launches run the
 *                     kernel for that grouping. */
typedef struct {
  int32_t max_tokens;       /* rows of Q/K/V/O the frame's launches address */
  int32_t max_seqs;
  int32_t max_blocks;       /* block-table entries of one pass */
  int32_t max_decode_items;
  int32_t max_chunk_tiles;
  int32_t max_combine_rows;
  int32_t max_parts;        /* partial-output slots of the workspace */
  int32_t packed_units;     /* 1: passes may hold short prompt chunks packed into decode
                               units (the decode variant with per-row limits runs for
                               every pass); 0: such passes are refused */
  int32_t chunk_items;      /* rbkv_chunk_items grouping of every pass's chunk tiles */
} rbkv_frame_caps;

/* Create a frame on the current device for passes of `cfg` (device memory for
 * the metadata and pinned host staging; the filled-in capacities are returned
 * in *caps_out when it is not NULL).  Errors: RBKV_ERR_INVALID (bad config or
 * max_tokens < 1), RBKV_ERR_UNSUPPORTED (shape off the fast kernels),
 * RBKV_ERR_CUDA. */
rbkv_status rbkv_frame_create(const rbkv_config* cfg, const rbkv_frame_caps* caps,
                              rbkv_frame** out, rbkv_frame_caps* caps_out);
void rbkv_frame_destroy(rbkv_frame* f);

/* Plan the pass for the frame's device and copy its metadata into the frame
 * on `stream` (from pinned staging; the host waits only when every staging
 * buffer is still in flight).  The pass must have the frame's config and fit
 * its capacities: RBKV_ERR_WORKSPACE names the capacity it exceeds (nothing is
 * changed; the plain entry points still serve that pass).  An empty pass is
 * loaded as zero counts. */
rbkv_status rbkv_frame_load(rbkv_frame* f, rbkv_pass* p, rbkv_stream stream);

/* rbkv_kv_append for the pass loaded last: k_new/v_new are [max_tokens][H_kv][D]
 * (rows past the pass's token count are not read). */
rbkv_status rbkv_frame_kv_append(rbkv_frame* f, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, rbkv_stream stream);

/* Workspace bytes rbkv_frame_attention needs (for max_parts partial slots). */
size_t rbkv_frame_workspace_bytes(const rbkv_frame* f);

/* rbkv_ragged_attention for the pass loaded last: q and o are [max_tokens][H_q][D]
 * (rows past the pass's token count are neither read as queries nor written);
 * workspace as rbkv_frame_workspace_bytes, 256-byte aligned. */
rbkv_status rbkv_frame_attention(rbkv_frame* f, const void* q, const void* k_cache,
                                 const void* v_cache, void* o, void* workspace,
                                 size_t workspace_bytes, rbkv_stream stream);

/* As rbkv_pass_device_status, for the frame's status word (sticky across the
 * passes loaded since it was last read). */
rbkv_status rbkv_frame_device_status(rbkv_frame* f, rbkv_stream stream);

/* ---- the rest of a decoder layer: tensor-core GEMM and RMSNorm --------------
 *
 * DeepSpeed-FastGen paper summary page, idea I1: a forward pass's latency
 * follows its token count; the token-proportional work of a layer besides
 * attention is its projections (QKV, output, the two MLP products) and the
 * normalisations around them.  These calls run those steps on the device, so
 * that a whole decoder layer can be put around the attention pass. */

typedef enum {
  RBKV_GEMM_PLAIN = 0,     /* C[m][n] = A B^T */
  RBKV_GEMM_RESIDUAL = 1,  /* C[m][n] = A B^T + R[m][n] */
  RBKV_GEMM_SWIGLU = 2     /* B's rows in blocks of 256: 128 gate rows, then the 128 up
                              rows of the same outputs; C[m][n/2] = silu(gate) * up with
                              output j of block b at column 128 b + j */
} rbkv_gemm_epilogue;

/* Device workspace that rbkv_gemm_bf16 / rbkv_gemm_bf16_qkv can use for a
 * product of this size: when its 128 x 256 output tiles are fewer than the
 * SMs (few rows: a weight-streaming product), K is split into pieces run by
 * different SMs, their fp32 partial sums kept here and added by a second
 * kernel that applies the epilogue.  0 when the product does not split. */
size_t rbkv_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k);

/* C = A . B^T in bf16 with fp32 accumulation on the tensor cores (tcgen05),
 * with a fused epilogue (rbkv_gemm_epilogue).  a: [m][k] row-major (the
 * activations); b: [n][k] row-major (a weight stored [out][in]); c: [m][n]
 * ([m][n/2] for RBKV_GEMM_SWIGLU); residual: [m][n] or NULL.  Device
 * pointers, 16-byte aligned; k a multiple of 8; n a multiple of 32 (256 for
 * SwiGLU); c must not overlap a or b (it may be the residual itself).
 * workspace: NULL, or device memory of workspace_bytes (256-byte aligned,
 * owned by the caller, not used by other work until this call's kernels end):
 * with at least rbkv_gemm_workspace_bytes(m, n, k) bytes the product may
 * split K (results then differ only by fp32 rounding order).
 * status: NULL or a device array of 4 int32 (code, wait site, index, block)
 * that a bounded wait that gives up writes, as a pass's status words.
 * Launches on `stream`.  Errors: RBKV_ERR_INVALID, RBKV_ERR_CUDA. */
rbkv_status rbkv_gemm_bf16(const void* a, const void* b, void* c, int64_t m, int64_t n, int64_t k,
                           const void* residual, int32_t epilogue, void* workspace,
                           size_t workspace_bytes, int32_t* status, rbkv_stream stream);

/* The QKV projection as one GEMM whose outputs are the attention pass's
 * inputs: w_qkv is [n_q + 2 n_kv][k] (the Q rows, then K, then V); q receives
 * [m][n_q], k_out and v_out [m][n_kv] (Q [T][H_q][D] and K_new, V_new
 * [T][H_kv][D] for n_q = H_q D, n_kv = H_kv D).  n_q and n_kv multiples of
 * 32; otherwise as rbkv_gemm_bf16. */
rbkv_status rbkv_gemm_bf16_qkv(const void* a, const void* w_qkv, void* q, void* k_out,
                               void* v_out, int64_t m, int64_t n_q, int64_t n_kv, int64_t k,
                               void* workspace, size_t workspace_bytes, int32_t* status,
                               rbkv_stream stream);

/* y[i][:] = x[i][:] / sqrt(mean_j x[i][j]^2 + eps) * weight[:] for m rows of
 * `hidden` bf16 values (fp32 arithmetic, bf16 out); hidden a multiple of 8,
 * 16-byte aligned device pointers.  Errors: RBKV_ERR_INVALID, RBKV_ERR_CUDA. */
rbkv_status rbkv_rmsnorm_bf16(const void* x, const void* weight, void* y, int64_t m,
                              int64_t hidden, float eps, rbkv_stream stream);

/* ---- measurement ----------------------------------------------------------- */

/* Kernel kinds for rbkv_profile_read. */
typedef enum {
  RBKV_KERNEL_KV_APPEND = 0,
  RBKV_KERNEL_CHUNK = 1,      /* tcgen05 prompt-chunk attention */
  RBKV_KERNEL_DECODE = 2,     /* split-KV decode attention (TMA + tensor cores) */
  RBKV_KERNEL_GENERIC = 3,    /* CUDA-core attention */
  RBKV_KERNEL_COMBINE = 4,    /* log-sum-exp combine */
  RBKV_KERNEL_META_UPLOAD = 5, /* a pass's metadata, host to device */
  RBKV_KERNEL_KINDS = 6
} rbkv_kernel_kind;

/* Kernels this process has launched through the library so far. */
int64_t rbkv_kernel_launches(void);

/* Turn per-launch CUDA-event timing on (1) or off (0).  While on, every kernel
 * launch is bracketed by two events recorded on its own stream. */
void rbkv_profile_enable(int32_t on);

/* Wait for the recorded events and return the summed device time (ms) and the
 * number of timed launches of one kernel kind since the last reset. */
rbkv_status rbkv_profile_read(int32_t kind, double* total_ms, int64_t* launches);

/* Forget all recorded launches. */
void rbkv_profile_reset(void);

#ifdef __cplusplus
}
#endif

#endif /* RBKV_H */
