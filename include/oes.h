/*
 * oes.h -- offloaded expert slots: the C ABI of the offloaded-MoE layer
 * forward over a GPU slot cache, for one NVIDIA GB300 (sm_103a).
 *
 * The path (FreeToken PR #676, Solution: the demand-token prefill):
 * a chunk is routed top-k; its distinct experts, a sorted list of fixed
 * length, are admitted into an LRU (or LRFU) slot cache in queries of at most
 * 128 ids; each query's misses are copied from a pinned-host expert source,
 * and no query evicts a slot an earlier query of the chunk touched; routes
 * are sorted into per-expert blocks (moe_align_block_size); the grouped
 * SwiGLU expert GEMM runs over the slot pool through an expert->slot remap
 * with its tiles sized by the layer's expert count, and it gives exactly the
 * bytes the same GEMM gives over the whole streamed layer.
 *
 * Conventions for every call:
 *   - Pointers are raw addresses.  "device" = GPU global memory; "host" =
 *     ordinary host memory; "mapped" = pinned host memory the GPU can read
 *     (cudaHostAlloc / cudaHostRegister; on GB300 any pinned allocation).
 *   - The caller allocates and owns every buffer.  The library owns only the
 *     small device tables (and the streams and events) behind the opaque
 *     handles oes_slot_cache, oes_expert_source and oes_stage_plan, created
 *     and destroyed explicitly, and the fixed scratch of
 *     moe_align_block_size_noalloc.
 *   - Calls are asynchronous on the given stream and never synchronise the
 *     host, except the *_load_state / *_read_state / *_read_lrfu /
 *     *_set_policy / *_create / *_destroy calls and oes_stage_plan_create,
 *     which say so.
 *   - The return value reports what the host can check before launching:
 *     OES_OK, OES_ERR_INVALID_ARG (null pointer, size out of range, buffer
 *     too small), OES_ERR_UNSUPPORTED (a size the library does not handle),
 *     OES_ERR_CAPACITY (a chunk the pool cannot hold), OES_ERR_CUDA (a CUDA
 *     call or launch failed; oes_last_error() has the message).  On any
 *     error nothing more is launched.
 *   - What only the GPU can see is OR-ed into a caller-provided device word
 *     `status` (OES_DEV_*), read by the caller at its own synchronisation.
 *     A kernel that finds a bad condition records it and skips the work
 *     that depends on it; it never traps.
 *   - Layouts are row-major and contiguous; all byte offsets are 64-bit.
 *   - bf16 / f16 values travel as uint16_t bit patterns.
 */
#ifndef OES_H
#define OES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *oes_stream_t; /* a cudaStream_t; NULL = legacy default stream */

enum {
  OES_OK = 0,
  OES_ERR_INVALID_ARG = 1,
  OES_ERR_UNSUPPORTED = 2,
  OES_ERR_CUDA = 3,
  OES_ERR_CAPACITY = 4
};

enum {
  OES_DEV_CAPACITY = 1, /* an ensure query had more misses than evictable slots */
  OES_DEV_BAD_ID = 2,   /* an id out of range, or a query not strictly ascending */
  OES_DEV_TIMEOUT = 4   /* a bounded wait gave up */
};

/* Expert formats.  NVFP4 weights are decoded exactly to f16 in shared memory
 * and the activations stay 16-bit (W4A16).  NVFP4_W4A4 uses the same expert
 * rows but also quantises the activations to NVFP4, under the maximum of the
 * layer's input scales (FreeToken PR #676, Solution and Tests: the W4A4
 * path takes the layer's scales, never another slot's).  x per 16 along H and
 * the SwiGLU output h per 16 along I become e2m1 codes with e4m3 block
 * scales: s = amax / (6 a), q = v / (sf a) in fp32, each rounded to nearest
 * even and saturating.  The GEMMs multiply the exact f16 products q * sf and
 * scale their fp32 sums by a and the weights' global scale, which is what a
 * block-scaled FP4 MMA computes, up to summation order.  It needs the view's
 * input_scale13 / input_scale2 (positive; a non-positive maximum sets
 * OES_DEV_BAD_ID and uses 1). */
enum { OES_WFMT_BF16 = 0, OES_WFMT_NVFP4 = 1, OES_WFMT_NVFP4_W4A4 = 2 };

/* Eviction policies of the slot cache.  LRU is the pages' (FreeToken PR #676,
 * the author's reply: the cache is LRU only).  LRFU is the scored policy the
 * pages name without a formula (one author's build admits by LRFU;
 * gdevenyi's review comment: a scored policy must pin a chunk's earlier
 * queries against its later ones).  It follows Lee et al. (IEEE Trans.
 * Computers 2001) with F(x) = (1 - 2^-k)^x in Q32.32 fixed point: each ensure
 * decays every slot's score once (score -= score >> k; k = 0 never decays,
 * which is LFU), evicts the non-hit, unpinned slots of smallest (score, slot),
 * empty slots first, adds 1.0 to each hit, starts each fill at 1.0, and
 * saturates at 2^51 - 1 units. */
enum { OES_POLICY_LRU = 0, OES_POLICY_LRFU = 1 };
#define OES_LRFU_MAX_K 18

#define OES_QUERY_MAX 128   /* ids per ensure query (FreeToken PR #676, Solution) */
#define OES_MAX_TOPK 32
#define OES_MAX_EXPERTS 4096
#define OES_MAX_SLOTS 8192

/* Capacity of moe_align_block_size's sorted_ids for R routes, E experts and
 * block size B: R + min(E, R) * (B - 1), rounded up to a multiple of B.  No
 * routing needs more.  block_expert holds OES_ALIGN_CAPACITY / B entries. */
#define OES_ALIGN_CAPACITY(R, E, B) \
  ((((int64_t)(R) + (int64_t)((E) < (R) ? (E) : (R)) * ((B) - 1)) + (B) - 1) / (B) * (B))

/* Message of the last error on this thread (static storage). */
const char *oes_last_error(void);

/* ------------------------------------------------------------------ route */

/* Router logits of the tiny workload: logits[t, e] = sum_h x[t, h] * gate[h, e]
 * with bf16 inputs and fp32 sums (the workload's "router logits from a bf16
 * gate").  x: device [T, H] bf16; gate: device [H, E] bf16; logits: device
 * [T, E] fp32.  1 <= T, 1 <= H, 1 <= E <= OES_MAX_EXPERTS. */
int moe_gate_logits(const uint16_t *x, const uint16_t *gate, int T, int H, int E, float *logits,
                    oes_stream_t stream);

/* Router logit types of moe_route_topk. */
enum { OES_LOGITS_F32 = 0, OES_LOGITS_BF16 = 1 };

/* Top-k routing (FreeToken PR #676, Problem and Solution: each token routes
 * to k experts; the workloads fix softmax-renormalised top-k).  For each
 * token t: ids[t, 0..k-1] = the k largest logits[t, :] in descending order,
 * ties to the lower expert id; weights[t, j] = softmax over the k selected
 * logits (equal to the full softmax renormalised over the top k).
 * logits: device [T, E] of `dtype` (OES_LOGITS_F32, or OES_LOGITS_BF16 as
 * uint16_t bit patterns, widened exactly to fp32 before any comparison); a
 * NaN logit ranks as -inf (then by id), -0 as +0; ids: device [T, k] int32;
 * weights: device [T, k] fp32.  1 <= k <= min(E, OES_MAX_TOPK),
 * E <= OES_MAX_EXPERTS. */
int moe_route_topk(const void *logits, int dtype, int T, int E, int k, int32_t *ids,
                   float *weights, oes_stream_t stream);

/* The chunk's distinct experts as a sorted list of fixed length (FreeToken
 * PR #676, Solution: the list's length does not depend on the routing, so
 * the host never waits on the device to size it).  distinct: device [min(R, E)] int32, ascending, padded at the tail
 * with -1; d_count: device [1] int32 = number of distinct experts.  ids out
 * of [0, E) are ignored.  ids: device [R] int32, R >= 0. */
int moe_distinct_experts(const int32_t *ids, int R, int E, int32_t *distinct, int32_t *d_count,
                         oes_stream_t stream);

/* ------------------------------------------------------------- slot cache */

/* An LRU cache of S slots shared by L layers of E experts each, keyed by
 * key = layer * E + expert (vLLM fork PR #48, What: one bank keyed by
 * (layer, expert)).  Device tables: map [L*E] (slot of each key or -1),
 * slot_key [S] (key of each slot or -1), slot_ts [S] (timestamp of the query
 * that last touched the slot; 0 = empty), a clock (last timestamp handed
 * out), counters hits / misses / evictions and decode_freq [L*E].
 * The slot pool itself (S rows of expert bytes) belongs to the caller.
 * A handle also owns the two side streams and the events of
 * moe_layer_forward_slots.  Calls on one handle are ordered by the caller:
 * they must not overlap in time from different host threads, and their
 * device work follows the order of the streams they are given (the tables
 * are one state).  Different handles are independent. */
typedef struct oes_slot_cache oes_slot_cache;

/* Allocates the tables (cudaMalloc, synchronous) on the current device and
 * sets every slot empty.  1 <= S <= OES_MAX_SLOTS, 1 <= E <= OES_MAX_EXPERTS,
 * L >= 1, L * E < 2^31. */
int slot_cache_create(int S, int L, int E, oes_slot_cache **out);
/* Waits for the handle's two side streams, then frees its tables, streams and
 * events.  Work the caller queued on its own streams that uses the handle must
 * have finished (or be synchronised) first.  A null handle is a no-op. */
int slot_cache_destroy(oes_slot_cache *cache);

/* Replaces the state: slot_key / slot_ts host [S] (slot_ts 0 for an empty
 * slot, in [1, clock] otherwise), clock = last timestamp handed out, below
 * 2^47; rebuilds map, zeroes the counters.  Synchronous. */
int slot_cache_load_state(oes_slot_cache *cache, const int32_t *slot_key, const int64_t *slot_ts,
                          int64_t clock);

/* Puts the handle back in the state slot_cache_create leaves: every slot
 * empty, clock 0, counters, decode frequencies, LRFU scores, pins and the
 * chunk tag counter zero.  The policy stays as set.  Three memsets on
 * `stream`, ordered after the handle's earlier calls on it; no host
 * synchronisation, so a graph may capture it. */
int slot_cache_reset(oes_slot_cache *cache, oes_stream_t stream);

/* Copies the state to host arrays (any may be NULL): map [L*E], slot_key
 * [S], slot_ts [S], clock [1], counters [3] = hits, misses, evictions,
 * decode_freq [L*E].  Synchronises `stream` first. */
int slot_cache_read_state(const oes_slot_cache *cache, int32_t *map, int32_t *slot_key,
                          int64_t *slot_ts, int64_t *clock, int64_t *counters,
                          int64_t *decode_freq, oes_stream_t stream);

/* Bytes of the cache's device tables, and asynchronous device-to-device
 * copies of them (one small kernel): snapshot saves every table (map, slots,
 * timestamps, clock, counters, decode_freq, LRFU scores and pins, the chunk
 * tag counter) into dst, restore puts such a snapshot back.  dst / src:
 * 16-byte aligned device buffers of slot_cache_state_bytes() bytes (a
 * multiple of 16).  Used to replay a query sequence from a known state
 * without a host sync. */
size_t slot_cache_state_bytes(const oes_slot_cache *cache);
int slot_cache_snapshot(const oes_slot_cache *cache, void *dst, oes_stream_t stream);
int slot_cache_restore(oes_slot_cache *cache, const void *src, oes_stream_t stream);

/* Device pointer to the layer's expert->slot remap: map + layer * E, [E]
 * int32, the slot of each of the layer's experts or -1 (vLLM fork PR #48,
 * What: the remap from logical expert to physical row).  Valid until slot_cache_destroy. */
int slot_cache_layer_map(const oes_slot_cache *cache, int layer, const int32_t **e2s);

/* One LRU ensure query (FreeToken PR #676, Solution: the distinct experts
 * go to lru_ensure in queries of at most 128; the author's reply: LRU only).
 * experts: device [n] int32, the query's experts of `layer`, strictly
 * ascending, -1 entries ignored; n <= OES_QUERY_MAX.
 * Effect: one clock tick; every hit slot and every filled slot gets the new
 * timestamp; the i-th smallest missing key takes the i-th victim, victims
 * being the slots the query does not hit in order (empty first, then
 * ascending (timestamp, slot)); an evicted key leaves the map.
 * miss: device [3 * OES_QUERY_MAX] int32, entry i = (key, slot, evicted key
 * or -1) for i < *n_miss; n_miss: device [1] int32.
 * record_stats = 0 (demand admission): hits / misses / evictions /
 * decode_freq are not touched (FreeToken PR #676, Solution: a prefill's
 * admissions count neither as decode frequency nor in the LRU stats); 1:
 * they grow, and
 * decode_freq[key] += 1 for every key of the query.
 * Device status: OES_DEV_BAD_ID (id out of range or not ascending) or
 * OES_DEV_CAPACITY (more misses than non-hit slots): nothing changes and
 * *n_miss = 0.  A query with no valid id is a no-op. */
int slot_cache_ensure(oes_slot_cache *cache, int layer, const int32_t *experts, int n,
                      int record_stats, int32_t *miss, int32_t *n_miss, int32_t *status,
                      oes_stream_t stream);

/* slot_cache_ensure with a pin tag.  Under LRFU, a nonzero tag excludes from
 * the victims every slot pinned to it and pins every slot the query touches,
 * so the queries of one chunk, sharing a tag, never evict one another's
 * slots.  Under LRU the tag is ignored (LRU already takes those slots last).
 * tag > 0 is used as given; OES_TAG_NEW_CHUNK draws the next tag from a
 * counter in the cache's device tables (1, 2, ...; reset by load_state and
 * set_policy, part of a snapshot) and OES_TAG_SAME_CHUNK reuses the last
 * one drawn, so a chunk replayed from a CUDA graph still gets a fresh tag.
 * moe_layer_forward_slots passes OES_TAG_NEW_CHUNK for its first query and
 * OES_TAG_SAME_CHUNK for the others. */
#define OES_TAG_NEW_CHUNK (-1)
#define OES_TAG_SAME_CHUNK (-2)
int slot_cache_ensure_tagged(oes_slot_cache *cache, int layer, const int32_t *experts, int n,
                             int record_stats, int32_t tag, int32_t *miss, int32_t *n_miss,
                             int32_t *status, oes_stream_t stream);

/* Selects the eviction policy (OES_POLICY_LRU, the default, or
 * OES_POLICY_LRFU with decay shift k in [0, OES_LRFU_MAX_K]).  Waits for the
 * device, then gives every occupied slot the score 1.0 and clears the pins.
 * slot_cache_load_state does the same reset and keeps the policy; snapshot
 * and restore include scores and pins. */
int slot_cache_set_policy(oes_slot_cache *cache, int policy, int lrfu_k);

/* Copies the LRFU scores (host [S] uint64, Q32.32) and pins (host [S] int32)
 * out; either may be NULL.  Synchronises `stream` first. */
int slot_cache_read_lrfu(const oes_slot_cache *cache, uint64_t *crf, int32_t *pin,
                         oes_stream_t stream);

/* Where the experts live on the host: L layers of E rows of row_bytes each;
 * layer l's rows start at the mapped address layer_base[l] (several layers
 * may share one buffer).  row_bytes is a multiple of 16; bases are 16-byte
 * aligned.  Create/destroy allocate/free a small device table. */
typedef struct oes_expert_source oes_expert_source;
int oes_expert_source_create(const void *const *layer_base, int L, int E, int64_t row_bytes,
                             oes_expert_source **out);
int oes_expert_source_destroy(oes_expert_source *src);

/* Copies each miss of one query from the host source into its slot
 * (FreeToken PR #676, Solution: a query's misses land before the following
 * query may evict anything; vLLM fork PR #48, What: the rows move by a
 * kernel with a fixed grid that reads the mapped host memory directly).  For i < *n_miss (read on the
 * device; at most max_misses): pool[slot] <- source row of key, the whole
 * row (weights, scales and per-expert scalars).  pool: device [S, row_bytes]
 * with the source's row_bytes.  Rows not named by the miss list are not
 * written.  Device status OES_DEV_BAD_ID for a key or slot out of range. */
int slot_cache_copy_misses(const oes_expert_source *src, void *pool, int S, const int32_t *miss,
                           const int32_t *n_miss, int max_misses, int32_t *status,
                           oes_stream_t stream);

/* Copies all E rows of one layer into a contiguous device buffer (the
 * whole-layer stream of FreeToken PR #676, Problem), with the miss copies'
 * SM-load kernel (one warp per SM) rather than a DMA copy.
 * dst: device [E, row_bytes], 16-byte aligned. */
int oes_copy_layer(const oes_expert_source *src, int layer, void *dst, oes_stream_t stream);

/* ------------------------------------------------------------------ align */

/* moe_align_block_size (FreeToken PR #676, Solution and Tests: correct past
 * 1024 experts, each route placed exactly once and only in one of its own
 * expert's blocks; vLLM
 * fork PR #48, What: logical alignment, ignore_invalid_experts).  A stable
 * counting sort of routes r = 0..R-1 by expert ids[r]:
 *   sorted_ids: device [OES_ALIGN_CAPACITY(R, E, B)] int32: experts in
 *     ascending order, each expert's routes in ascending r, padded to a
 *     multiple of B with the value R; every entry past the last block = R;
 *   block_expert: device [OES_ALIGN_CAPACITY / B] int32: expert of each
 *     block, -1 past the last block;
 *   n_post_pad: device [1] int32: used entries (a multiple of B).
 * Experts with no route get no block.  ids outside [0, E) are skipped; with
 * ignore_invalid = 0 they also set OES_DEV_BAD_ID.
 * workspace: device scratch of moe_align_workspace_size(R, E, B) bytes.
 * 0 <= R < 2^30, 1 <= E <= OES_MAX_EXPERTS, 1 <= B <= 1024. */
size_t moe_align_workspace_size(int R, int E, int B);
int moe_align_block_size(const int32_t *ids, int R, int E, int B, int ignore_invalid,
                         int32_t *sorted_ids, int32_t *block_expert, int32_t *n_post_pad,
                         int32_t *status, void *workspace, size_t workspace_bytes,
                         oes_stream_t stream);

/* moe_align_block_size without a workspace argument: the same result, with
 * its scratch in a fixed buffer inside the library.  The pages have no
 * counterpart; this is for callers that cannot call cudaMalloc on this path,
 * such as an engine that has handed all free GPU memory to its own pool, or a
 * caller that must not risk the device-wide synchronisation cudaMalloc and
 * cudaFree can cause in the middle of its work.
 * The buffer is OES_ALIGN_NOALLOC_SCRATCH_BYTES (1 MiB) of device memory on
 * every GPU that loads the library, held until the process exits.  A call
 * needing more scratch than that (moe_align_workspace_size(R, E, B)) returns
 * OES_ERR_INVALID_ARG and launches nothing; e.g. 40960 routes over 512
 * experts need 41 KB, 65536 routes over 2100 experts 269 KB.
 * The first call on a device looks the buffer's device address up
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  The call allocates nothing.
 * The address is kept per device ordinal for the life of the process: it
 * does not survive a reset of the device (cudaDeviceReset, or anything else
 * that destroys the primary context), after which this call must not be
 * used again in the process.
 * Every call on a device shares the one buffer, which keeps the last call's
 * contents; each call writes all the scratch it reads, so nothing has to
 * start at zero.  Calls whose kernels overlap on the GPU (other streams, or
 * other threads) race on the buffer and must be ordered by the caller.
 * Arguments, outputs and status as for moe_align_block_size. */
#define OES_ALIGN_NOALLOC_SCRATCH_BYTES (1 << 20)
int moe_align_block_size_noalloc(const int32_t *ids, int R, int E, int B, int ignore_invalid,
                                 int32_t *sorted_ids, int32_t *block_expert, int32_t *n_post_pad,
                                 int32_t *status, oes_stream_t stream);

/* ------------------------------------------------------------ expert GEMM */

/* The experts a chunk routes to, as the grouped GEMM sees them (FreeToken
 * PR #676, Solution: RoutedExperts; the view knows both the slot pool and
 * the layer, whose expert count and input scales it takes).  E is the LAYER's expert count and
 * alone sizes the tiles; S is only the pool's extent.
 * Expert row layout (row_bytes each, one per slot):
 *   bf16:  w13 [2I, H] bf16 (rows 0..I-1 gate, I..2I-1 up), w2 [H, I] bf16;
 *   nvfp4: w13 values [2I, H/2] u8 (e2m1 pairs, element 2i in the low
 *          nibble), w13 scales [H/64, 2I, 4] e4m3 (K-chunk-major), w2 values
 *          [H, I/2], w2 scales [I/64, H, 4], then fp32 gs13, gs2, in13, in2
 *          (global scales and input scales), each section 16-byte aligned.
 * Weights decode as e2m1 * e4m3 * gs. */
typedef struct {
  int layer;                  /* the layer, for the record */
  int E;                      /* the layer's expert count (sizes the tiles) */
  const int32_t *e2s;         /* device [E]: slot of each expert, -1 = not resident */
  int wfmt;                   /* OES_WFMT_BF16 or OES_WFMT_NVFP4 */
  const void *pool;           /* device base of the slot pool [S, row_bytes] */
  int64_t row_bytes;          /* bytes per slot row */
  int S;                      /* slots in the pool */
  int H, I;                   /* hidden and expert intermediate sizes */
  const float *input_scale13; /* device [E] or NULL: the layer's w13 input scales */
  const float *input_scale2;  /* device [E] or NULL: the layer's w2 input scales */
} oes_routed_experts;

/* Tile plan (FreeToken PR #676, Solution: nvfp4_moe.prefill_config sizes
 * the tiles by routes per expert of the layer, never per slot): the block
 * size B shared by moe_align_block_size and the GEMM, a function of R and
 * the layer's E only: 16 when ceil(R / E) <= 8 (the weight-major kernel,
 * 128 weight rows x 16 routes per MMA), else 128 (the token-major kernel,
 * 128 routes x 256 weight rows per MMA). */
int oes_tile_plan(int R, int E, int *block);

/* Workspace bytes of moe_grouped_gemm_slots for T tokens at top-k. */
size_t moe_grouped_gemm_workspace_size(const oes_routed_experts *view, int T, int k);

/* Device pointers to the GEMM's intermediates inside its workspace, for
 * checking the steps: h [capacity, I] (16-bit: bf16 for bf16 weights, f16
 * otherwise; for W4A4 the quantised q * sf), y [T*k, H] bf16, and x16 [T, H]
 * f16, the 16-bit copy of x the NVFP4 GEMMs read (for W4A4, q * sf of the
 * quantised x; NULL for bf16 weights).  Any output may be NULL. */
int moe_grouped_gemm_workspace_views(const oes_routed_experts *view, int T, int k,
                                     void *workspace, uint16_t **h, uint16_t **y,
                                     uint16_t **x16);

/* The grouped SwiGLU expert GEMM over the slot pool (FreeToken PR #676,
 * Solution: a demand chunk reuses the decode GEMM, reading each expert at
 * its slot, and must match the streamed layer byte for byte).  For
 * every block b < n_post_pad / B of expert e = block_expert[b], with
 * weights at slot e2s[e]:
 *   h = silu(x_r @ gate^T) * (x_r @ up^T), y_r = h @ w2^T    (fp32 sums)
 * for the routes r in sorted_ids[b*B .. b*B+B) (padding skipped), then
 *   out[t] = sum_{j=0..k-1} weights[t, j] * y_{t*k+j}         (j in order)
 * rounded to bf16; h and y are held as 16-bit values in the workspace.
 * NVFP4 weights are decoded exactly and the global scales applied to the
 * fp32 sums.  Every reduction order depends only on the routing, never on
 * the slots, so the result over the pool equals the result over a
 * contiguous layer buffer (e2s = identity) bit for bit.  When the GEMM1
 * tiles of the largest routing of T x k fill at most half the SMs (one-token
 * decode), each tile's K range is summed in two halves on two SMs, added in
 * fp32 in a fixed order (half 0 + half 1) before the SwiGLU.
 * x: device [T, H] bf16; ids / weights: the router's [T, k] int32 / fp32
 * (a route whose id is outside [0, E) contributes nothing); sorted_ids,
 * block_expert, n_post_pad: moe_align_block_size with B from oes_tile_plan
 * (anything else is OES_ERR_INVALID_ARG); out: device [T, H] bf16.
 * A routed expert with e2s < 0 sets OES_DEV_BAD_ID and its routes give 0.
 * H, I multiples of 64 in [64, 16384]. */
int moe_grouped_gemm_slots(const oes_routed_experts *view, const uint16_t *x, int T, int k,
                           const int32_t *ids, const float *weights, const int32_t *sorted_ids,
                           const int32_t *block_expert, const int32_t *n_post_pad, int B,
                           void *workspace, size_t workspace_bytes, uint16_t *out,
                           int32_t *status, oes_stream_t stream);

/* --------------------------------------------------------- whole layer */

/* One chunk of one layer, as the composite calls see it. */
typedef struct {
  const float *logits;    /* device [T, E] fp32, or NULL to compute them from x and gate */
  const uint16_t *gate;   /* device [H, E] bf16 when logits is NULL */
  const uint16_t *x;      /* device [T, H] bf16 */
  int T, k;
  uint16_t *out;          /* device [T, H] bf16 */
  int32_t *status;        /* device [1] int32, OR-ed */
  void *workspace;        /* device scratch of moe_layer_workspace_size() bytes, 256-aligned */
  size_t workspace_bytes;
} oes_chunk;

/* The layer as stored: expert count, sizes, weight format and the layer's
 * input scales (device [E] each, or NULL). */
typedef struct {
  int E, H, I, wfmt;
  const float *input_scale13;
  const float *input_scale2;
} oes_layer_desc;

size_t moe_layer_workspace_size(const oes_layer_desc *layer, int T, int k);

/* Device pointers to the router's outputs and the align outputs inside a
 * layer workspace (for checking the steps of a composite call): ids [T*k],
 * weights [T*k], distinct [min(T*k, E)] and its count, sorted_ids, block_expert,
 * n_post_pad.  Any output pointer may be NULL. */
int moe_layer_workspace_views(const oes_layer_desc *layer, int T, int k, void *workspace,
                              int32_t **ids, float **weights, int32_t **distinct,
                              int32_t **d_count, int32_t **sorted_ids, int32_t **block_expert,
                              int32_t **n_post_pad);

/* The slot path, stream-ordered on `stream` with no host synchronisation
 * (FreeToken PR #676, Solution): route (or gate logits + route) -> distinct
 * experts -> the queries of OES_QUERY_MAX distinct experts, each ensured
 * (record_stats as given) in order -> align -> grouped GEMM over `pool`
 * through the layer's remap -> combine.  The number of queries is
 * ceil(min(T*k, E) / OES_QUERY_MAX), known on the host.
 * Schedule: each query's misses are copied on `stream`, in query order,
 * after that query's ensure.  The cache's side stream runs the later
 * ensures, the expert groups and then the GEMM over the experts that were
 * hits; a second side stream runs the align (right after routing) and the
 * GEMM over each query's copied experts once they are in.  A query of more
 * than 32 ids copies its misses in two launches (the last min(n/2, 16) of
 * its n misses second), each part with its own GEMM, so that after the last
 * copy at most 16 experts' GEMM remains.  A chunk of one query and at most
 * 1024 routes (a decode step) takes a shorter schedule with the same
 * results: routing, distinct experts, the ensure, the expert groups and the
 * align in one kernel on `stream`, the GEMM over the hits right behind it
 * on `stream`, the copies on the side stream and the GEMM over the copied
 * experts on the second side stream.  The later ensures may run before
 * earlier copies finish: ensure reads no pool bytes, and with the chunk
 * fitting the pool no query evicts a slot an earlier query touched, so the
 * tables, the slots written and the bytes are those of ensuring and
 * copying query by query.
 * The pool must hold every expert the chunk needs at once (the author's
 * reply on FreeToken PR #676): with min(T*k, E) > S this returns
 * OES_ERR_CAPACITY and launches nothing; the caller streams the layer.
 * The call makes no host synchronisation and no allocation, and its side
 * streams fork from and join `stream` through events.  So a decode step
 * (record_stats = 1) can be captured from `stream` into a CUDA graph and
 * replayed on new tokens written into the same x / logits buffers.  The
 * first call with a given shape sets one-time kernel attributes, so run it
 * once before capturing. */
int moe_layer_forward_slots(oes_slot_cache *cache, const oes_expert_source *src, void *pool,
                            int layer, const oes_layer_desc *desc, const oes_chunk *chunk,
                            int record_stats, oes_stream_t stream);

/* The whole-layer streamed path, the baseline the slot path must equal
 * (FreeToken PR #676, Problem: every expert of the layer is streamed for the
 * chunk): copy all E rows of `layer` into layer_buf (device [E, row_bytes])
 * on copy_stream, route and align on compute_stream meanwhile, then run the
 * same grouped GEMM over layer_buf with the identity remap once the copy is
 * done.  The copy waits for the work queued on compute_stream before the
 * call (an earlier GEMM over the same buffer).  copy_stream may equal
 * compute_stream. */
int moe_layer_forward_stream(const oes_expert_source *src, void *layer_buf, int layer,
                             const oes_layer_desc *desc, const oes_chunk *chunk,
                             oes_stream_t copy_stream, oes_stream_t compute_stream);

/* Demand-token dispatch (FreeToken PR #676, Solution and Tests).  A
 * threshold N (0 = off, the default) sends prefill chunks of up to N tokens
 * through the slot cache as decode does; longer chunks stream the whole
 * layer.  Returns 1 when a chunk of T tokens at top-k over E experts takes the
 * slot path of an S-slot pool: 0 < T <= demand_tokens and min(T*k, E) <= S
 * (a chunk needing more distinct experts than the pool holds streams, since a
 * later query would evict a slot the chunk still reads); else 0.  Host only,
 * no CUDA call. */
int oes_takes_slot_path(int T, int k, int E, int S, int demand_tokens);

/* One layer forward with the demand-token dispatch: the slot path
 * (moe_layer_forward_slots on `stream`) when oes_takes_slot_path() says so,
 * else the whole-layer streamed path (moe_layer_forward_stream, copying on
 * copy_stream into layer_buf).  *took_slots (host, may be NULL) reports the
 * choice.  Both paths give the same bytes for the same chunk. */
int moe_layer_forward(oes_slot_cache *cache, const oes_expert_source *src, void *pool,
                      void *layer_buf, int layer, const oes_layer_desc *desc,
                      const oes_chunk *chunk, int demand_tokens, int record_stats,
                      oes_stream_t copy_stream, oes_stream_t stream, int *took_slots);

/* ------------------------------------------------- staged layer sequence */

/* Prefill staging over a sequence of layers (vLLM fork PR #51, Details,
 * "Prefill staging"): two device buffers of one whole layer each alternate
 * by layer; the rows of layer i+1 are copied on a copy stream while layer i
 * computes, ordered by events (the pages copy by DMA; here the miss copies'
 * one-warp-per-SM kernel, which holds the host link's rate where DMA falls
 * back over tens of GB of pinned source); at the start of the step the
 * placement tables are read back once and each layer's non-resident experts
 * become contiguous runs.  Resident experts are read from their slots and
 * their rows are never written.
 *
 * Pool layout for the staged runner: one allocation of S + 2E rows of
 * row_bytes.  Rows 0..S-1 are the cache's slots; rows S + b*E + e
 * (b = 0, 1) are staging buffer b, expert e at its own row, so one 3-D
 * tensor map and one remap serve both kinds of expert and the GEMM is the
 * very kernel of the slot and streamed paths.
 *
 * oes_stage_plan_create: layers host [n] (each in [0, L), repeats allowed).
 * skip_resident = 1: an expert with a slot is read from it and not copied;
 * 0: every expert of the layer is copied (the whole-layer stream, with
 * prefetch).  Reads the cache's map back with one host synchronisation of
 * `stream` (work queued there before the call is part of the placement the
 * plan sees), allocates the plan's device remap [n][E] and its events.  The
 * plan describes the cache as it is now: it is valid until the next call
 * that changes the cache (ensure, load_state, restore). */
typedef struct oes_stage_plan oes_stage_plan;
int oes_stage_plan_create(const oes_slot_cache *cache, const int *layers, int n, int skip_resident,
                          oes_stream_t stream, oes_stage_plan **out);
int oes_stage_plan_destroy(oes_stage_plan *plan);

/* Layer i of the plan: *n_runs runs [runs[2j], runs[2j+1]) of staged
 * experts, ascending and maximal (runs: host [2*E] or NULL), *rows = the
 * staged experts in all. */
int oes_stage_plan_layer(const oes_stage_plan *plan, int i, int *n_runs, int32_t *runs, int *rows);

/* Forwards the plan's n layers in order: layer i = plan layer i with chunk
 * chunks[i] (host array [n]; chunks run one after another on
 * compute_stream, so they may share x, out and workspace).  Per layer: the
 * copy kernel moves the runs into staging buffer i % 2 on copy_stream (after the
 * compute of layer i-2 released that buffer, and after all work queued on
 * compute_stream before the call), then on compute_stream route -> align
 * -> wait for the copies -> grouped GEMM -> combine, with the plan's remap.
 * Each chunk's output equals moe_layer_forward_stream's for that layer and
 * chunk, byte for byte.  pool: device [S + 2E, row_bytes] as above.  The
 * first call with a given source row size builds the plan's device copy
 * tables (an allocation and a synchronous upload).  The
 * plan's events order the copies, so one plan feeds one runner at a time;
 * oes_stage_plan_destroy waits for the last runner's compute to finish. */
int moe_layers_forward_staged(const oes_stage_plan *plan, const oes_expert_source *src, void *pool,
                              const oes_layer_desc *desc, const oes_chunk *chunks,
                              oes_stream_t copy_stream, oes_stream_t compute_stream);

#ifdef __cplusplus
}
#endif

#endif /* OES_H */
