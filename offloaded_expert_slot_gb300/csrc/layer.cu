// The whole-layer composites: the slot path and the streamed path, each a
// stream-ordered sequence of the library's own calls with no host sync.
//
// FreeToken PR #676, Solution: a prefill chunk loads the experts it routes
// to into the slot cache, in queries of 128 distinct experts, each query's
// misses copied before the next, then runs the same grouped GEMM over the
// slot pool at their slots; Problem: the streamed path copies every expert
// of the layer for the chunk.
#include <algorithm>

#include "common.cuh"
#include "gemm_types.h"
#include "internal.h"

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
  uint8_t* resident;  // [E] expert resident before the chunk
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
  w.miss = static_cast<int32_t*>(take(3 * OES_QUERY_MAX * 4));
  w.n_miss = static_cast<int32_t*>(take(4));
  w.sorted_ids = static_cast<int32_t*>(take((size_t)std::max<int64_t>(cap, 1) * 4));
  w.block_expert = static_cast<int32_t*>(take((size_t)std::max<int64_t>(cap / B, 1) * 4));
  w.n_post_pad = static_cast<int32_t*>(take(4));
  w.e2s_identity = static_cast<int32_t*>(take((size_t)E * 4));
  w.resident = static_cast<uint8_t*>(take((size_t)E));
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

// resident[e] = 1 for the chunk's experts that already have a slot.  Taken
// before the first ensure: a layer never routes to more experts than the pool
// holds, so no query of the chunk evicts a slot the chunk uses, and these
// experts keep their slots (and bytes) through all of the chunk's queries.
__global__ void resident_flags_kernel(const int32_t* __restrict__ distinct, int n, int E, int layer,
                                      const int32_t* __restrict__ map, uint8_t* __restrict__ resident) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) resident[e] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = distinct[i];
    if (e >= 0 && e < E) resident[e] = map[(int64_t)layer * E + e] >= 0 ? 1 : 0;
  }
}

__global__ void iota_kernel(int32_t* a, int n) {
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
  return moe_route_topk(logits, c->T, d->E, c->k, w.ids, w.w, s);
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
  if ((rc = route(d, c, w, stream))) return rc;
  if ((rc = moe_distinct_experts(w.ids, R, E, w.distinct, w.d_count, stream))) return rc;
  const int Lq = std::min(R, E);
  resident_flags_kernel<<<1, 1024, 0, stream>>>(w.distinct, Lq, E, layer, cache->map, w.resident);
  OES_CHECK_LAUNCH("resident_flags_kernel");
  if ((rc = moe_align_block_size(w.ids, R, E, B, 1, w.sorted_ids, w.block_expert, w.n_post_pad,
                                 c->status, w.align_ws, w.align_bytes, stream)))
    return rc;
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
                         w.gemm_bytes, c->status, stream, &g)))
    return rc;
  // side stream: the GEMM over the experts already resident, overlapping the
  // copies of the misses on the caller's stream
  OES_TRY_CUDA(cudaEventRecord(cache->fork, stream));
  OES_TRY_CUDA(cudaStreamWaitEvent(cache->side, cache->fork, 0));
  if ((rc = gemm_run(g, 1, w.resident, cache->side))) return rc;
  OES_TRY_CUDA(cudaEventRecord(cache->join, cache->side));
  // caller's stream: each query of at most OES_QUERY_MAX distinct experts is
  // ensured and its misses copied before the next query
  for (int q0 = 0; q0 < Lq; q0 += OES_QUERY_MAX) {
    const int n = std::min(OES_QUERY_MAX, Lq - q0);
    if ((rc = slot_cache_ensure(cache, layer, w.distinct + q0, n, record_stats, w.miss, w.n_miss,
                                c->status, stream)))
      return rc;
    if ((rc = slot_cache_copy_misses(src, pool, cache->S, w.miss, w.n_miss, n, c->status, stream)))
      return rc;
  }
  if ((rc = gemm_run(g, 2, w.resident, stream))) return rc;   // the experts just copied
  OES_TRY_CUDA(cudaStreamWaitEvent(stream, cache->join, 0));
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
  if ((rc = oes_copy_layer(src, layer, layer_buf, copy_stream))) return rc;
  cudaEvent_t copied = nullptr;
  if (copy_stream != compute_stream) {
    OES_TRY_CUDA(cudaEventCreateWithFlags(&copied, cudaEventDisableTiming));
    OES_TRY_CUDA(cudaEventRecord(copied, copy_stream));
  }
  iota_kernel<<<ceil_div(E, 256), 256, 0, compute_stream>>>(w.e2s_identity, E);
  OES_CHECK_LAUNCH("iota_kernel");
  if ((rc = route(d, c, w, compute_stream))) return rc;
  if ((rc = moe_align_block_size(w.ids, R, E, B, 1, w.sorted_ids, w.block_expert, w.n_post_pad,
                                 c->status, w.align_ws, w.align_bytes, compute_stream)))
    return rc;
  if (copied) {
    OES_TRY_CUDA(cudaStreamWaitEvent(compute_stream, copied, 0));
    OES_TRY_CUDA(cudaEventDestroy(copied));
  }
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
  return moe_grouped_gemm_slots(&v, c->x, T, k, w.ids, w.w, w.sorted_ids, w.block_expert,
                                w.n_post_pad, B, w.gemm_ws, w.gemm_bytes, c->out, c->status,
                                compute_stream);
}
