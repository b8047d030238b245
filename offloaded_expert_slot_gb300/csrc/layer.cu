// The whole-layer composites: the slot path and the streamed path, each a
// stream-ordered sequence of the library's own calls with no host sync.
//
// FreeToken PR #676, Solution: a short prefill chunk fills the slot cache
// with just its routed experts, 128 distinct experts per query with every
// query's copies done before the next query, and then reuses the decode
// GEMM over the slots; Problem: streaming moves all of the layer's experts
// for every chunk.
#include <cuda_fp16.h>

#include <algorithm>
#include <climits>
#include <utility>
#include <vector>

#include "align_dev.cuh"
#include "common.cuh"
#include "ensure_dev.cuh"
#include "gemm_types.h"
#include "internal.h"
#include "route_dev.cuh"

namespace oes {
namespace {

struct LayerWs {
  float* logits;
  int32_t* ids;
  float* w;
  int32_t* distinct;
  int32_t* d_count;
  int32_t* miss;
  int32_t* n_miss;
  int32_t* sorted_ids;
  int32_t* block_expert;
  int32_t* n_post_pad;
  int32_t* e2s_identity;
  uint8_t* resident;  // [E] group of each of the chunk's experts (hit, or missed in query q)
  int32_t* gcount;    // [kGroups] experts in each group
  void* align_ws;
  size_t align_bytes;
  void* gemm_ws;
  size_t gemm_bytes;
  size_t total;
};

LayerWs carve_layer(void* base, const oes_layer_desc* d, int T, int k) {
  LayerWs w{};
  const int R = T * k, E = d->E;
  const int B = tile_plan(R, E);
  const int64_t cap = OES_ALIGN_CAPACITY(R, E, B);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    void* r = p + off;
    off += up(bytes);
    return r;
  };
  w.logits = static_cast<float*>(take((size_t)T * E * 4));
  w.ids = static_cast<int32_t*>(take((size_t)R * 4));
  w.w = static_cast<float*>(take((size_t)R * 4));
  w.distinct = static_cast<int32_t*>(take((size_t)std::max(1, std::min(R, E)) * 4));
  w.d_count = static_cast<int32_t*>(take(4));
  const int Q = std::max(1, (std::min(R, E) + OES_QUERY_MAX - 1) / OES_QUERY_MAX);
  w.miss = static_cast<int32_t*>(take((size_t)Q * 3 * OES_QUERY_MAX * 4));
  w.n_miss = static_cast<int32_t*>(take((size_t)Q * 4));
  w.sorted_ids = static_cast<int32_t*>(take((size_t)std::max<int64_t>(cap, 1) * 4));
  w.block_expert = static_cast<int32_t*>(take((size_t)std::max<int64_t>(cap / B, 1) * 4));
  w.n_post_pad = static_cast<int32_t*>(take(4));
  w.e2s_identity = static_cast<int32_t*>(take((size_t)E * 4));
  w.resident = static_cast<uint8_t*>(take((size_t)E));
  w.gcount = static_cast<int32_t*>(take((size_t)kGroups * 4));
  w.align_bytes = moe_align_workspace_size(R, E, B);
  w.align_ws = take(w.align_bytes);
  oes_routed_experts v{};
  v.E = E;
  v.H = d->H;
  v.I = d->I;
  v.wfmt = d->wfmt;
  w.gemm_bytes = moe_grouped_gemm_workspace_size(&v, T, k);
  w.gemm_ws = take(w.gemm_bytes);
  w.total = off + 256;
  return w;
}

// group[e] of the chunk's experts, taken after every query of the chunk has
// been ensured: kGroupHit for an expert that was a hit in its own query,
// kGroupMiss0 + 2q + p for one that query q missed, p = 0 or 1 the part of
// the query's misses its copy belongs to (miss_split; 0 for experts not in
// the chunk).  A hit keeps its slot and bytes to the end of the chunk: its query
// gives it a newer timestamp than any slot no query of the chunk has
// touched, and since the pool holds all of the chunk's experts at once
// (checked up front) every later query finds enough such older slots to
// evict.  An expert resident before the chunk but belonging to a later query
// has no such guarantee: an earlier query may evict it, and it is then a
// miss of its own query like any other.

__device__ __forceinline__ void group_flags_cta(const int32_t* distinct, int n, int E, int layer,
                                                const int32_t* miss, const int32_t* n_miss, int Q,
                                                uint8_t* group, int32_t* __restrict__ gcount) {
  __shared__ int32_t cnt[kGroups];
  for (int e = threadIdx.x; e < E; e += blockDim.x) group[e] = 0;
  for (int g = threadIdx.x; g < kGroups; g += blockDim.x) cnt[g] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = distinct[i];
    if (e >= 0 && e < E) group[e] = kGroupHit;
  }
  __syncthreads();
  for (int q = 0; q < Q; ++q) {
    const int m = min(n_miss[q], OES_QUERY_MAX);
    const int nq = min(OES_QUERY_MAX, n - q * OES_QUERY_MAX);
    const int split = nq > kSplitIds ? miss_split(m) : m;
    for (int i = threadIdx.x; i < m; i += blockDim.x) {
      const int e = miss[(q * OES_QUERY_MAX + i) * 3] - layer * E;
      if (e >= 0 && e < E) group[e] = (uint8_t)(kGroupMiss0 + 2 * q + (i >= split));
    }
  }
  // experts per group: a filtered GEMM launch over an empty group returns
  // before it deals out units
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int g = group[e];
    if (g) atomicAdd(&cnt[g], 1);
  }
  __syncthreads();
  for (int g = threadIdx.x; g < kGroups; g += blockDim.x) gcount[g] = cnt[g];
}

__global__ void group_flags_kernel(const int32_t* __restrict__ distinct, int n, int E, int layer,
                                   const int32_t* __restrict__ miss,
                                   const int32_t* __restrict__ n_miss, int Q,
                                   uint8_t* __restrict__ group, int32_t* __restrict__ gcount) {
  pdl_begin();
  group_flags_cta(distinct, n, E, layer, miss, n_miss, Q, group, gcount);
}

// The front of a small chunk's slot path in one launch of two CTAs (at most
// kSmallR routes, one ensure query, E <= kFrontMaxExperts): route, distinct
// experts, the query's ensure, the expert groups, the align and, for NVFP4
// weights, the f16 copy of x -- the device code of the separate kernels, so
// every table and output is the same bit for bit.  A decode step's chain of
// six launches and two cross-stream waits becomes one launch.
constexpr int kFrontMaxExperts = 1024;
struct FrontArgs {
  const float* logits;
  int T, k, E, H, layer, record_stats, B, nzero;
  int64_t cap;
  CacheView c;
  int32_t *ids, *distinct, *d_count, *miss, *n_miss, *gcount, *sorted_ids, *block_expert,
      *n_post_pad, *zero, *status;
  float* w;
  uint8_t* group;
  const uint16_t* x;  // [T, H] bf16
  uint16_t* x16;      // [T, H] its f16 copy (NVFP4 weights), or null
};

template <int EPL>
__global__ void __launch_bounds__(kEnsureThreads) decode_front_kernel(const FrontArgs a) {
  pdl_begin();
  extern __shared__ uint64_t dsm[];  // each step's own scratch, in turn
  // what one step hands the next stays in shared memory; the global copies
  // the later kernels read are written at the end
  __shared__ int32_t s_ids[kSmallR];
  __shared__ float s_w[kSmallR];
  __shared__ int32_t s_distinct[OES_QUERY_MAX];
  __shared__ int32_t s_miss[3 * OES_QUERY_MAX];
  __shared__ int32_t s_dcount, s_nmiss;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
  const int R = a.T * a.k, Lq = min(R, a.E);
  // both CTAs route (the same routes, bit for bit); CTA 0 then asks the
  // cache and sets the groups while CTA 1 aligns the routes and converts x
  // (the threshold filter up to 512 experts; past that its 32 logits a lane
  // would spill at this kernel's 64 registers a thread)
  for (int t = warp; t < a.T; t += kEnsureThreads / 32) {
    if constexpr (EPL <= 16)
      topk_row_filtered<1, EPL, float>(a.logits + (size_t)t * a.E, a.E, a.k, lane, s_ids + t * a.k,
                                       s_w + t * a.k, reinterpret_cast<uint2*>(dsm) + 33 * warp);
    else
      topk_row<EPL, float>(a.logits + (size_t)t * a.E, a.E, a.k, lane, s_ids + t * a.k, s_w + t * a.k);
  }
  __syncthreads();
  if (blockIdx.x == 1) {
    align_small_cta(s_ids, R, a.E, a.B, a.cap, 1, a.sorted_ids, a.block_expert, a.n_post_pad,
                    a.status, a.zero, a.nzero, reinterpret_cast<int32_t*>(dsm));
    if (a.x16) {
      const int64_t n = (int64_t)a.T * a.H;
      for (int64_t i = tid; i < n; i += nt) {
        const float f = __uint_as_float(static_cast<uint32_t>(a.x[i]) << 16);
        a.x16[i] = __half_as_ushort(__float2half_rn(f));
      }
    }
    return;
  }
  for (int i = tid; i < R; i += nt) {
    a.ids[i] = s_ids[i];
    a.w[i] = s_w[i];
  }
  for (int e = tid; e < a.E; e += nt) a.group[e] = 0;
  distinct_cta(s_ids, R, a.E, s_distinct, &s_dcount, reinterpret_cast<uint8_t*>(dsm));
  __syncthreads();
  ensure_query(a.c, a.layer, s_distinct, Lq, a.record_stats, OES_TAG_NEW_CHUNK, s_miss, &s_nmiss,
               a.status, dsm);
  __syncthreads();
  // the groups of one query (group_flags_cta with Q = 1): every distinct
  // expert a hit, then each miss its part; the counts follow from D and the
  // misses (each miss is one of the D experts)
  const int D = s_dcount, m = min(s_nmiss, OES_QUERY_MAX);
  const int split = Lq > kSplitIds ? miss_split(m) : m;
  for (int i = tid; i < Lq; i += nt) {
    const int e = s_distinct[i];
    a.distinct[i] = e;
    if (e >= 0 && e < a.E) a.group[e] = kGroupHit;
  }
  for (int i = tid; i < 3 * m; i += nt) a.miss[i] = s_miss[i];
  for (int g = tid; g < kGroups; g += nt)
    a.gcount[g] = g == kGroupHit ? D - m : g == kGroupMiss0 ? split : g == kGroupMiss0 + 1 ? m - split : 0;
  if (tid == 0) {
    *a.d_count = D;
    *a.n_miss = s_nmiss;
  }
  __syncthreads();  // the hits' group bytes before the misses' overwrite them
  for (int i = tid; i < m; i += nt) {
    const int e = s_miss[3 * i] - a.layer * a.E;
    if (e >= 0 && e < a.E) a.group[e] = (uint8_t)(kGroupMiss0 + (i >= split));
  }
}

__global__ void iota_kernel(int32_t* a, int n) {
  pdl_begin();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) a[i] = i;
}

int check_chunk(const oes_layer_desc* d, const oes_chunk* c) {
  OES_REQUIRE(d && c, "layer forward: null desc or chunk");
  OES_REQUIRE(d->E >= 1 && d->E <= OES_MAX_EXPERTS, "layer forward: bad E=%d", d->E);
  OES_REQUIRE(c->x && c->out && c->workspace && (c->logits || c->gate),
              "layer forward: chunk needs x, out, workspace and logits or gate");
  OES_REQUIRE(c->T >= 0 && c->k >= 1 && c->k <= OES_MAX_TOPK && c->k <= d->E,
              "layer forward: bad T=%d k=%d", c->T, c->k);
  OES_REQUIRE(((uintptr_t)c->workspace & 255) == 0, "layer forward: workspace not 256-byte aligned");
  const size_t need = moe_layer_workspace_size(d, c->T, c->k);
  OES_REQUIRE(c->workspace_bytes >= need, "layer forward: workspace %zu < %zu bytes",
              c->workspace_bytes, need);
  return OES_OK;
}

// route -> (ids, weights) in the workspace
int route(const oes_layer_desc* d, const oes_chunk* c, const LayerWs& w, cudaStream_t s) {
  const float* logits = c->logits;
  if (!logits) {
    int rc = moe_gate_logits(c->x, c->gate, c->T, d->H, d->E, w.logits, s);
    if (rc) return rc;
    logits = w.logits;
  }
  return moe_route_topk(logits, OES_LOGITS_F32, c->T, d->E, c->k, w.ids, w.w, s);
}

}  // namespace
}  // namespace oes

using namespace oes;

extern "C" size_t moe_layer_workspace_size(const oes_layer_desc* d, int T, int k) {
  if (!d || T < 0 || k < 1 || d->E < 1) return 0;
  return carve_layer(nullptr, d, T, k).total;
}

extern "C" int moe_layer_workspace_views(const oes_layer_desc* d, int T, int k, void* workspace,
                                         int32_t** ids, float** weights, int32_t** distinct,
                                         int32_t** d_count, int32_t** sorted_ids,
                                         int32_t** block_expert, int32_t** n_post_pad) {
  OES_REQUIRE(d && workspace && T >= 0 && k >= 1 && d->E >= 1, "moe_layer_workspace_views: bad arguments");
  const LayerWs w = carve_layer(workspace, d, T, k);
  if (ids) *ids = w.ids;
  if (weights) *weights = w.w;
  if (distinct) *distinct = w.distinct;
  if (d_count) *d_count = w.d_count;
  if (sorted_ids) *sorted_ids = w.sorted_ids;
  if (block_expert) *block_expert = w.block_expert;
  if (n_post_pad) *n_post_pad = w.n_post_pad;
  return OES_OK;
}

extern "C" int moe_layer_forward_slots(oes_slot_cache* cache, const oes_expert_source* src, void* pool,
                                       int layer, const oes_layer_desc* d, const oes_chunk* c,
                                       int record_stats, oes_stream_t stream) {
  int rc = check_chunk(d, c);
  if (rc) return rc;
  OES_REQUIRE(cache && src && pool, "moe_layer_forward_slots: null cache, source or pool");
  OES_REQUIRE(cache->E == d->E && src->E == d->E && src->L == cache->L,
              "moe_layer_forward_slots: cache, source and layer disagree on L/E");
  OES_REQUIRE(layer >= 0 && layer < cache->L, "moe_layer_forward_slots: layer %d out of range", layer);
  const int T = c->T, k = c->k, E = d->E, R = T * k;
  if (std::min(R, E) > cache->S) {
    set_error("moe_layer_forward_slots: the chunk may route to %d experts, more than the %d slots",
              std::min(R, E), cache->S);
    return OES_ERR_CAPACITY;
  }
  if (T == 0) return OES_OK;
  const LayerWs w = carve_layer(c->workspace, d, T, k);
  const int B = tile_plan(R, E);
  const int Lq = std::min(R, E);
  const int Q = (Lq + OES_QUERY_MAX - 1) / OES_QUERY_MAX;
  cudaStream_t side = cache->side;
  auto miss_of = [&](int q) { return w.miss + (size_t)q * 3 * OES_QUERY_MAX; };
  // the chunk's pin tag, drawn on the device by its first query: its
  // queries never evict one another's slots under a scored policy (LRU
  // ignores it), also when the call is replayed from a CUDA graph
  auto query = [&](int q, cudaStream_t s) {
    const int n = std::min(OES_QUERY_MAX, Lq - q * OES_QUERY_MAX);
    return slot_cache_ensure_tagged(cache, layer, w.distinct + q * OES_QUERY_MAX, n, record_stats,
                                    q == 0 ? OES_TAG_NEW_CHUNK : OES_TAG_SAME_CHUNK, miss_of(q),
                                    w.n_miss + q, c->status, s);
  };
  auto copy = [&](int q, int part, cudaStream_t s) {
    const int n = std::min(OES_QUERY_MAX, Lq - q * OES_QUERY_MAX);
    return copy_misses_part(src, pool, cache->S, miss_of(q), w.n_miss + q, n, part, c->status, s);
  };
  // the GEMM is validated and its parameters built before anything is
  // launched: a call that fails here leaves the cache as it was
  oes_routed_experts v{};
  v.layer = layer;
  v.E = E;
  v.e2s = cache->map + (size_t)layer * E;
  v.wfmt = d->wfmt;
  v.pool = pool;
  v.row_bytes = src->row_bytes;
  v.S = cache->S;
  v.H = d->H;
  v.I = d->I;
  v.input_scale13 = d->input_scale13;
  v.input_scale2 = d->input_scale2;
  GemmPlan g;
  if ((rc = gemm_prepare(&v, c->x, T, k, w.sorted_ids, w.block_expert, w.n_post_pad, B, w.gemm_ws,
                         w.gemm_bytes, c->status, &g)))
    return rc;
  if (R <= kSmallR && Q == 1 && E <= kFrontMaxExperts) {
    // A small chunk (a decode step): the front in one launch, then the GEMM
    // over the hits right behind it on the caller's stream; the query's
    // copies on the side stream and each part's copied experts on the gemm
    // stream, as below.
    if (g.a4 && (rc = gemm_prepare_x(g, stream))) return rc;
    const float* logits = c->logits;
    if (!logits) {
      if ((rc = moe_gate_logits(c->x, c->gate, T, d->H, E, w.logits, stream))) return rc;
      logits = w.logits;
    }
    const GemmCounters sc = gemm_counters(g);
    FrontArgs a{};
    a.logits = logits;
    a.T = T;
    a.k = k;
    a.E = E;
    a.H = d->H;
    a.layer = layer;
    a.record_stats = record_stats;
    a.B = B;
    a.cap = OES_ALIGN_CAPACITY(R, E, B);
    a.c = view_of(cache);
    a.ids = w.ids;
    a.w = w.w;
    a.distinct = w.distinct;
    a.d_count = w.d_count;
    a.miss = miss_of(0);
    a.n_miss = w.n_miss;
    a.group = w.resident;
    a.gcount = w.gcount;
    a.sorted_ids = w.sorted_ids;
    a.block_expert = w.block_expert;
    a.n_post_pad = w.n_post_pad;
    a.zero = sc.ptr;
    a.nzero = sc.n;
    a.status = c->status;
    a.x = c->x;
    a.x16 = (g.wf && !g.a4) ? g.x16 : nullptr;
    int spad = 2;
    while (spad < cache->S) spad <<= 1;
    const size_t smem =
        std::max({(size_t)E, (size_t)spad * 8, ((size_t)2 * E + (size_t)std::max(R, 1)) * 4,
                  (size_t)kEnsureThreads / 32 * 33 * sizeof(uint2)});
    const void* fn = E <= 512 ? reinterpret_cast<const void*>(decode_front_kernel<16>)
                              : reinterpret_cast<const void*>(decode_front_kernel<32>);
    if ((rc = set_max_dynamic_smem(fn, smem, "decode_front_kernel: shared memory limit"))) return rc;
    if ((rc = prefer_max_shared_carveout(fn, "decode_front_kernel: carveout"))) return rc;
    if (E <= 512) launch_kernel(decode_front_kernel<16>, 2, kEnsureThreads, smem, stream, a);
    else launch_kernel(decode_front_kernel<32>, 2, kEnsureThreads, smem, stream, a);
    OES_CHECK_LAUNCH("decode_front_kernel");
    OES_TRY_CUDA(cudaEventRecord(cache->fork, stream));
    const int np = Lq > kSplitIds ? 2 : 1;
    OES_TRY_CUDA(cudaStreamWaitEvent(side, cache->fork, 0));
    for (int p = 0; p < np; ++p) {
      if ((rc = copy(0, np == 2 ? p : -1, side))) return rc;
      OES_TRY_CUDA(cudaEventRecord(cache->copied[p], side));
    }
    OES_TRY_CUDA(cudaEventRecord(cache->join, side));
    if ((rc = gemm_run(g, kGroupHit, w.resident, w.gcount, stream))) return rc;
    cudaStream_t gs = cache->gemm;
    for (int p = 0; p < np; ++p) {
      OES_TRY_CUDA(cudaStreamWaitEvent(gs, cache->copied[p], 0));
      if ((rc = gemm_run(g, kGroupMiss0 + p, w.resident, w.gcount, gs))) return rc;
    }
    OES_TRY_CUDA(cudaEventRecord(cache->gjoin, gs));
    OES_TRY_CUDA(cudaStreamWaitEvent(stream, cache->join, 0));
    OES_TRY_CUDA(cudaStreamWaitEvent(stream, cache->gjoin, 0));
    return gemm_combine(g, w.ids, w.w, c->out, stream);
  }
  // caller's stream: route, distinct experts, the first query
  if ((rc = route(d, c, w, stream))) return rc;
  OES_TRY_CUDA(cudaEventRecord(cache->routed, stream));
  if ((rc = moe_distinct_experts(w.ids, R, E, w.distinct, w.d_count, stream))) return rc;
  if ((rc = query(0, stream))) return rc;
  OES_TRY_CUDA(cudaEventRecord(cache->fork, stream));
  // gemm stream: the align and the GEMMs' x, which need only the routes, run
  // while the queries are ensured
  cudaStream_t gs = cache->gemm;
  OES_TRY_CUDA(cudaStreamWaitEvent(gs, cache->routed, 0));
  const GemmCounters sc = gemm_counters(g);
  if ((rc = align_run(w.ids, R, E, B, 1, w.sorted_ids, w.block_expert, w.n_post_pad, c->status,
                      w.align_ws, w.align_bytes, sc.ptr, sc.n, gs)))
    return rc;
  if ((rc = gemm_prepare_x(g, gs))) return rc;
  OES_TRY_CUDA(cudaEventRecord(cache->prepared, gs));
  // side stream: the later queries in order (ensure reads no pool bytes, and
  // with the chunk fitting the pool no query evicts a slot an earlier query
  // touched, so a query's copies may trail the later ensures), the expert
  // groups, then the GEMM over the hits once the align is done
  OES_TRY_CUDA(cudaStreamWaitEvent(side, cache->fork, 0));
  for (int q = 1; q < Q; ++q) {
    if ((rc = query(q, side))) return rc;
    OES_TRY_CUDA(cudaEventRecord(cache->ensured[q], side));
  }
  launch_kernel(group_flags_kernel, 1, 1024, 0, side, w.distinct, Lq, E, layer, w.miss, w.n_miss, Q,
                w.resident, w.gcount);
  OES_CHECK_LAUNCH("group_flags_kernel");
  OES_TRY_CUDA(cudaEventRecord(cache->flagged, side));
  OES_TRY_CUDA(cudaStreamWaitEvent(side, cache->prepared, 0));
  if ((rc = gemm_run(g, kGroupHit, w.resident, w.gcount, side))) return rc;
  OES_TRY_CUDA(cudaEventRecord(cache->join, side));
  // caller's stream: each query's misses in query order, each query's copies
  // after its own ensure, in two parts when it has more than kSplitIds ids;
  // each part's copied experts run once its copies are in, so that after the
  // last copy only the GEMM over the last part (at most 16 experts, or a
  // small query's misses) remains
  auto parts = [&](int q) {
    return std::min(OES_QUERY_MAX, Lq - q * OES_QUERY_MAX) > kSplitIds ? 2 : 1;
  };
  for (int q = 0; q < Q; ++q) {
    if (q > 0) OES_TRY_CUDA(cudaStreamWaitEvent(stream, cache->ensured[q], 0));
    for (int p = 0; p < parts(q); ++p) {
      if ((rc = copy(q, parts(q) == 2 ? p : -1, stream))) return rc;
      OES_TRY_CUDA(cudaEventRecord(cache->copied[2 * q + p], stream));
    }
  }
  // the gemm stream: each part's copied experts after the group flags and
  // that part's copies, beside the GEMM over the hits (empty parts, as in a
  // warm decode step, then cost the side stream nothing)
  OES_TRY_CUDA(cudaStreamWaitEvent(gs, cache->flagged, 0));
  for (int q = 0; q < Q; ++q) {
    for (int p = 0; p < parts(q); ++p) {
      OES_TRY_CUDA(cudaStreamWaitEvent(gs, cache->copied[2 * q + p], 0));
      if ((rc = gemm_run(g, kGroupMiss0 + 2 * q + p, w.resident, w.gcount, gs))) return rc;
    }
  }
  OES_TRY_CUDA(cudaEventRecord(cache->gjoin, gs));
  OES_TRY_CUDA(cudaStreamWaitEvent(stream, cache->join, 0));
  OES_TRY_CUDA(cudaStreamWaitEvent(stream, cache->gjoin, 0));
  return gemm_combine(g, w.ids, w.w, c->out, stream);
}

extern "C" int moe_layer_forward_stream(const oes_expert_source* src, void* layer_buf, int layer,
                                        const oes_layer_desc* d, const oes_chunk* c,
                                        oes_stream_t copy_stream, oes_stream_t compute_stream) {
  int rc = check_chunk(d, c);
  if (rc) return rc;
  OES_REQUIRE(src && layer_buf, "moe_layer_forward_stream: null source or layer buffer");
  OES_REQUIRE(src->E == d->E && layer >= 0 && layer < src->L, "moe_layer_forward_stream: bad layer");
  const int T = c->T, k = c->k, E = d->E, R = T * k;
  if (T == 0) return OES_OK;
  const LayerWs w = carve_layer(c->workspace, d, T, k);
  const int B = tile_plan(R, E);
  // the GEMM is validated before anything is launched
  oes_routed_experts v{};
  v.layer = layer;
  v.E = E;
  v.e2s = w.e2s_identity;
  v.wfmt = d->wfmt;
  v.pool = layer_buf;
  v.row_bytes = src->row_bytes;
  v.S = E;
  v.H = d->H;
  v.I = d->I;
  v.input_scale13 = d->input_scale13;
  v.input_scale2 = d->input_scale2;
  GemmPlan g;
  if ((rc = gemm_prepare(&v, c->x, T, k, w.sorted_ids, w.block_expert, w.n_post_pad, B, w.gemm_ws,
                         w.gemm_bytes, c->status, &g)))
    return rc;
  cudaEvent_t copied = nullptr;
  if (copy_stream != compute_stream) {
    // the copy overwrites layer_buf only after work queued earlier on
    // compute_stream (a previous layer's GEMM over the same buffer) is done
    cudaEvent_t entry = nullptr;
    OES_TRY_CUDA(cudaEventCreateWithFlags(&entry, cudaEventDisableTiming));
    OES_TRY_CUDA(cudaEventRecord(entry, compute_stream));
    OES_TRY_CUDA(cudaStreamWaitEvent(copy_stream, entry, 0));
    OES_TRY_CUDA(cudaEventDestroy(entry));
  }
  if ((rc = oes_copy_layer(src, layer, layer_buf, copy_stream))) return rc;
  if (copy_stream != compute_stream) {
    OES_TRY_CUDA(cudaEventCreateWithFlags(&copied, cudaEventDisableTiming));
    OES_TRY_CUDA(cudaEventRecord(copied, copy_stream));
  }
  launch_kernel(iota_kernel, ceil_div(E, 256), 256, 0, compute_stream, w.e2s_identity, E);
  OES_CHECK_LAUNCH("iota_kernel");
  if ((rc = route(d, c, w, compute_stream))) return rc;
  const GemmCounters sc = gemm_counters(g);
  if ((rc = align_run(w.ids, R, E, B, 1, w.sorted_ids, w.block_expert, w.n_post_pad, c->status,
                      w.align_ws, w.align_bytes, sc.ptr, sc.n, compute_stream)))
    return rc;
  if ((rc = gemm_prepare_x(g, compute_stream))) return rc;  // overlaps the layer copy
  if (copied) {
    OES_TRY_CUDA(cudaStreamWaitEvent(compute_stream, copied, 0));
    OES_TRY_CUDA(cudaEventDestroy(copied));
  }
  if ((rc = gemm_run(g, 0, nullptr, nullptr, compute_stream))) return rc;
  return gemm_combine(g, w.ids, w.w, c->out, compute_stream);
}

extern "C" int oes_takes_slot_path(int T, int k, int E, int S, int demand_tokens) {
  if (T <= 0 || demand_tokens <= 0 || T > demand_tokens) return 0;
  const int64_t R = (int64_t)T * k;
  return (R < E ? R : E) <= S ? 1 : 0;
}

extern "C" int moe_layer_forward(oes_slot_cache* cache, const oes_expert_source* src, void* pool,
                                 void* layer_buf, int layer, const oes_layer_desc* d,
                                 const oes_chunk* c, int demand_tokens, int record_stats,
                                 oes_stream_t copy_stream, oes_stream_t stream, int* took_slots) {
  OES_REQUIRE(d && c && cache, "moe_layer_forward: null desc, chunk or cache");
  const int slots = oes_takes_slot_path(c->T, c->k, d->E, cache->S, demand_tokens);
  if (took_slots) *took_slots = slots;
  if (slots) return moe_layer_forward_slots(cache, src, pool, layer, d, c, record_stats, stream);
  return moe_layer_forward_stream(src, layer_buf, layer, d, c, copy_stream, stream);
}

// ------------------------------------------------------------------ staging
// vLLM fork PR #51, Details ("Prefill staging"): whole-layer double buffer,
// next-layer prefetch on a side stream, contiguous non-resident runs
// from one placement readback per step.

struct oes_stage_plan {
  int n, S, L, E, device;
  std::vector<int> layers;
  std::vector<std::vector<std::pair<int, int>>> runs;  // [n] staged runs [e0, e1)
  std::vector<int> rows;                               // [n] staged experts
  int32_t* e2s;                                        // device [n][E]
  cudaEvent_t entry, copied[2], done[2];
  // the runs as copy-kernel tables, built by the first runner call for its
  // source's row size: layer i's runs are run_tab[run_first[i] ...]
  int64_t run_rb = 0;
  std::vector<CopyRun> run_host;
  std::vector<int> run_first, run_count;
  std::vector<int64_t> run_items;
  CopyRun* run_tab = nullptr;
};

namespace {

void destroy_plan(oes_stage_plan* p) {
  if (!p) return;
  cudaFree(p->e2s);
  cudaFree(p->run_tab);
  for (cudaEvent_t e : {p->entry, p->copied[0], p->copied[1], p->done[0], p->done[1]})
    if (e) cudaEventDestroy(e);
  delete p;
}

}  // namespace

extern "C" int oes_stage_plan_create(const oes_slot_cache* cache, const int* layers, int n,
                                     int skip_resident, oes_stream_t stream, oes_stage_plan** out) {
  OES_REQUIRE(cache && layers && out, "oes_stage_plan_create: null pointer");
  OES_REQUIRE(n >= 1 && n <= (1 << 16), "oes_stage_plan_create: bad layer count %d", n);
  const int L = cache->L, E = cache->E, S = cache->S;
  for (int i = 0; i < n; ++i)
    OES_REQUIRE(layers[i] >= 0 && layers[i] < L, "oes_stage_plan_create: layer %d out of range",
                layers[i]);
  std::vector<int32_t> map;
  if (skip_resident) {
    map.resize((size_t)L * E);
    OES_TRY_CUDA(cudaMemcpyAsync(map.data(), cache->map, map.size() * sizeof(int32_t),
                                 cudaMemcpyDeviceToHost, stream));
    OES_TRY_CUDA(cudaStreamSynchronize(stream));
  }
  auto* p = new oes_stage_plan();
  p->n = n;
  p->S = S;
  p->L = L;
  p->E = E;
  p->device = cache->device;
  p->layers.assign(layers, layers + n);
  p->runs.resize(n);
  p->rows.assign(n, 0);
  std::vector<int32_t> e2s((size_t)n * E);
  for (int i = 0; i < n; ++i) {
    const int32_t* m = skip_resident ? map.data() + (size_t)layers[i] * E : nullptr;
    const int32_t staged0 = S + (i & 1) * E;
    int e = 0;
    while (e < E) {
      if (m && m[e] >= 0) {
        e2s[(size_t)i * E + e] = m[e];
        ++e;
        continue;
      }
      const int e0 = e;
      while (e < E && !(m && m[e] >= 0)) {
        e2s[(size_t)i * E + e] = staged0 + e;
        ++e;
      }
      p->runs[i].emplace_back(e0, e);
      p->rows[i] += e - e0;
    }
  }
  cudaError_t err = cudaMalloc(&p->e2s, e2s.size() * sizeof(int32_t));
  if (err == cudaSuccess)
    err = cudaMemcpy(p->e2s, e2s.data(), e2s.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
  if (err == cudaSuccess) err = cudaEventCreateWithFlags(&p->entry, cudaEventDisableTiming);
  for (int b = 0; b < 2 && err == cudaSuccess; ++b) {
    err = cudaEventCreateWithFlags(&p->copied[b], cudaEventDisableTiming);
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&p->done[b], cudaEventDisableTiming);
  }
  if (err != cudaSuccess) {
    destroy_plan(p);
    return cuda_fail(err, "oes_stage_plan_create");
  }
  *out = p;
  return OES_OK;
}

extern "C" int oes_stage_plan_destroy(oes_stage_plan* p) {
  if (!p) return OES_OK;
  cudaError_t err = cudaEventSynchronize(p->done[0]);
  if (err == cudaSuccess) err = cudaEventSynchronize(p->done[1]);
  destroy_plan(p);
  if (err != cudaSuccess) return cuda_fail(err, "oes_stage_plan_destroy");
  return OES_OK;
}

extern "C" int oes_stage_plan_layer(const oes_stage_plan* p, int i, int* n_runs, int32_t* runs,
                                    int* rows) {
  OES_REQUIRE(p && i >= 0 && i < p->n, "oes_stage_plan_layer: bad plan or index");
  const auto& r = p->runs[i];
  if (n_runs) *n_runs = (int)r.size();
  if (rows) *rows = p->rows[i];
  if (runs)
    for (size_t j = 0; j < r.size(); ++j) {
      runs[2 * j] = r[j].first;
      runs[2 * j + 1] = r[j].second;
    }
  return OES_OK;
}

extern "C" int moe_layers_forward_staged(const oes_stage_plan* p, const oes_expert_source* src,
                                         void* pool, const oes_layer_desc* d,
                                         const oes_chunk* chunks, oes_stream_t copy_stream,
                                         oes_stream_t compute_stream) {
  OES_REQUIRE(p && src && pool && d && chunks, "moe_layers_forward_staged: null pointer");
  OES_REQUIRE(src->L == p->L && src->E == p->E && d->E == p->E,
              "moe_layers_forward_staged: source, plan and layer disagree on L or E");
  OES_REQUIRE(((uintptr_t)pool & 15) == 0, "moe_layers_forward_staged: pool not 16-byte aligned");
  for (int i = 0; i < p->n; ++i) {
    int rc = check_chunk(d, &chunks[i]);
    if (rc) return rc;
  }
  const PlainLaunches plain;  // no programmatic launches in the staged sequence
  const int E = p->E;
  const int64_t rb = src->row_bytes;
  uint8_t* base = static_cast<uint8_t*>(pool);
  // every layer's GEMM is validated and prepared before anything is launched
  std::vector<GemmPlan> plans(p->n);
  for (int i = 0; i < p->n; ++i) {
    const oes_chunk* c = &chunks[i];
    if (c->T == 0) continue;
    const LayerWs w = carve_layer(c->workspace, d, c->T, c->k);
    oes_routed_experts v{};
    v.layer = p->layers[i];
    v.E = E;
    v.e2s = p->e2s + (size_t)i * E;
    v.wfmt = d->wfmt;
    v.pool = pool;
    v.row_bytes = rb;
    v.S = p->S + 2 * E;
    v.H = d->H;
    v.I = d->I;
    v.input_scale13 = d->input_scale13;
    v.input_scale2 = d->input_scale2;
    const int rc = gemm_prepare(&v, c->x, c->T, c->k, w.sorted_ids, w.block_expert, w.n_post_pad,
                                tile_plan(c->T * c->k, E), w.gemm_ws, w.gemm_bytes, c->status,
                                &plans[i]);
    if (rc) return rc;
  }
  auto* mp = const_cast<oes_stage_plan*>(p);  // the run tables are a cache of the plan
  if (mp->run_rb != rb) {
    mp->run_host.clear();
    mp->run_first.assign(p->n, 0);
    mp->run_count.assign(p->n, 0);
    mp->run_items.assign(p->n, 0);
    for (int i = 0; i < p->n; ++i) {
      const int b = i & 1;
      int64_t items = 0;
      mp->run_first[i] = (int)mp->run_host.size();
      for (const auto& r : p->runs[i]) {
        const int64_t bytes = (int64_t)(r.second - r.first) * rb;
        mp->run_host.push_back(CopyRun{(int64_t)r.first * rb,
                                       ((int64_t)p->S + (int64_t)b * E + r.first) * rb, bytes, items});
        items += copy_run_items(bytes);
      }
      mp->run_count[i] = (int)p->runs[i].size();
      mp->run_items[i] = items;
    }
    cudaFree(mp->run_tab);
    mp->run_tab = nullptr;
    if (!mp->run_host.empty()) {
      OES_TRY_CUDA(cudaMalloc(&mp->run_tab, mp->run_host.size() * sizeof(CopyRun)));
      OES_TRY_CUDA(cudaMemcpy(mp->run_tab, mp->run_host.data(), mp->run_host.size() * sizeof(CopyRun),
                              cudaMemcpyHostToDevice));
    }
    mp->run_rb = rb;
  }
  OES_TRY_CUDA(cudaEventRecord(p->entry, compute_stream));
  OES_TRY_CUDA(cudaStreamWaitEvent(copy_stream, p->entry, 0));
  for (int i = 0; i < p->n; ++i) {
    const int b = i & 1, layer = p->layers[i];
    const oes_chunk* c = &chunks[i];
    // copy stream: this layer's runs into staging buffer b once layer i-2 let go of it
    if (i >= 2) OES_TRY_CUDA(cudaStreamWaitEvent(copy_stream, p->done[b], 0));
    if (p->run_count[i] > 0) {
      const int rc = launch_copy_runs(src->host_bases[layer], base, p->run_tab + p->run_first[i],
                                      p->run_count[i], 0, 0, 0, p->run_items[i], copy_stream);
      if (rc) return rc;
    }
    OES_TRY_CUDA(cudaEventRecord(p->copied[b], copy_stream));
    // compute stream: route and align overlap the copies; the GEMM waits for them
    const int T = c->T, k = c->k, R = T * k;
    if (T > 0) {
      const LayerWs w = carve_layer(c->workspace, d, T, k);
      const int B = tile_plan(R, E);
      int rc = route(d, c, w, compute_stream);
      const GemmCounters sc = gemm_counters(plans[i]);
      if (!rc)
        rc = align_run(w.ids, R, E, B, 1, w.sorted_ids, w.block_expert, w.n_post_pad, c->status,
                       w.align_ws, w.align_bytes, sc.ptr, sc.n, compute_stream);
      if (!rc) rc = gemm_prepare_x(plans[i], compute_stream);
      if (rc) return rc;
      OES_TRY_CUDA(cudaStreamWaitEvent(compute_stream, p->copied[b], 0));
      if ((rc = gemm_run(plans[i], 0, nullptr, nullptr, compute_stream))) return rc;
      if ((rc = gemm_combine(plans[i], w.ids, w.w, c->out, compute_stream))) return rc;
    } else {
      OES_TRY_CUDA(cudaStreamWaitEvent(compute_stream, p->copied[b], 0));
    }
    OES_TRY_CUDA(cudaEventRecord(p->done[b], compute_stream));
  }
  return OES_OK;
}
