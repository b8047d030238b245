// The LRU slot cache (tables in GPU memory, updated without a host sync),
// the pinned-host expert source, and the miss-row copies.
//
// FreeToken PR #676, Solution: the distinct experts reach lru_ensure in
// queries of at most 128, a query's misses land before the following query
// may evict, and a prefill's admissions count neither as decode frequency
// nor in the LRU statistics.  The author's reply on that page: LRU only.
// vLLM fork PR #48, What: all MoE layers share one bank, keyed by
// (layer, expert), and the rows move by a fixed-grid kernel that reads the
// mapped host memory directly.
#include <algorithm>
#include <climits>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "ensure_dev.cuh"

namespace oes {
namespace {

// One ensure query in one CTA (ensure_query).
__global__ void __launch_bounds__(kEnsureThreads)
    ensure_kernel(CacheView c, int layer, const int32_t* __restrict__ experts, int n,
                  int record_stats, int tag, int spad, int32_t* __restrict__ miss,
                  int32_t* __restrict__ n_miss, int32_t* __restrict__ status) {
  pdl_begin();
  extern __shared__ uint64_t skey[];  // [spad]
  ensure_query(c, layer, experts, n, record_stats, tag, miss, n_miss, status, skey);
}

constexpr int kCopyThreads = 32;
constexpr int kCopyUnroll = 8;

// Fixed grid of one warp per SM: work item = (miss i, 4 KB chunk of its
// row).  Each lane moves 8 x 16 bytes per item, all eight loads issued
// before the stores.  4 KB in flight per SM (0.6 MB over the GPU) keeps the
// NVLink-C2C host link full (99% of a pinned DMA copy on a GB300), while
// the kernels the slot path runs beside the copies (the later queries'
// ensures, the GEMM over the hits) keep their speed: with 32 KB in flight
// per SM their loads queued behind the copy's host reads and ran 4-10x
// slower.
__global__ void __launch_bounds__(kCopyThreads)
    copy_misses_kernel(const uint8_t* const* __restrict__ bases, int L, int E, int64_t row_bytes,
                       uint8_t* __restrict__ pool, int S, const int32_t* __restrict__ miss,
                       const int32_t* __restrict__ n_miss_p, int max_misses, int part,
                       int32_t* __restrict__ status) {
  pdl_wait();
  const int nm = min(*n_miss_p, max_misses);
  // part 0 / 1: the misses before / from miss_split(nm); -1: all of them
  const int i0 = part == 1 ? miss_split(nm) : 0, i1 = part == 0 ? miss_split(nm) : nm;
  const int64_t vecs = row_bytes >> 4;
  const int64_t chunk = (int64_t)kCopyThreads * kCopyUnroll;
  const int64_t per_row = (vecs + chunk - 1) / chunk;
  const int64_t total = (int64_t)(i1 - i0) * per_row;
  for (int64_t it = blockIdx.x; it < total; it += gridDim.x) {
    const int i = i0 + static_cast<int>(it / per_row);
    const int64_t c0 = (it % per_row) * chunk;
    const int key = miss[3 * i], slot = miss[3 * i + 1];
    if (key < 0 || key >= L * E || slot < 0 || slot >= S) {
      if (threadIdx.x == 0 && c0 == 0) set_status(status, OES_DEV_BAD_ID);
      continue;
    }
    const uint4* src =
        reinterpret_cast<const uint4*>(bases[key / E] + (int64_t)(key % E) * row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(pool + (int64_t)slot * row_bytes);
    uint4 buf[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t v = c0 + u * kCopyThreads + threadIdx.x;
      if (v < vecs) buf[u] = __ldcs(src + v);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t v = c0 + u * kCopyThreads + threadIdx.x;
      if (v < vecs) dst[v] = buf[u];
    }
  }
}

// Contiguous host runs to device, with copy_misses_kernel's access pattern
// (one warp per SM, 4 KB per item, eight 16-byte loads a lane in flight):
// over this pool's host link SM loads keep their rate where DMA copies lose
// up to a fifth of it once the pinned source spans tens of GB.  Runs from
// `runs` (device [nruns]) or, when it is null, the single run `one`.
__global__ void __launch_bounds__(kCopyThreads)
    copy_runs_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                     const CopyRun* __restrict__ runs, int nruns, CopyRun one, int64_t nitems) {
  pdl_wait();
  const int64_t chunk = (int64_t)kCopyThreads * kCopyUnroll;  // 16-byte vectors per item
  for (int64_t it = blockIdx.x; it < nitems; it += gridDim.x) {
    CopyRun r = one;
    if (runs) {
      int lo = 0, hi = nruns - 1;  // last run whose first item <= it
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (runs[mid].item0 <= it) lo = mid;
        else hi = mid - 1;
      }
      r = runs[lo];
    }
    const int64_t vecs = r.bytes >> 4;
    const int64_t c0 = (it - r.item0) * chunk;
    const uint4* s4 = reinterpret_cast<const uint4*>(src + r.src_off);
    uint4* d4 = reinterpret_cast<uint4*>(dst + r.dst_off);
    uint4 buf[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t v = c0 + u * kCopyThreads + threadIdx.x;
      if (v < vecs) buf[u] = __ldcs(s4 + v);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t v = c0 + u * kCopyThreads + threadIdx.x;
      if (v < vecs) d4[v] = buf[u];
    }
  }
}

// Device-to-device copy of the cache's tables (snapshot / restore): a few
// tens of KB, where a kernel launch beats a copy-engine transfer.
__global__ void copy_tables_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                   int64_t n16) {
  pdl_begin();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

int copy_tables(const void* src, void* dst, size_t bytes, cudaStream_t stream) {
  OES_REQUIRE((((uintptr_t)src | (uintptr_t)dst) & 15) == 0 && bytes % 16 == 0,
              "slot cache snapshot/restore: buffers must be 16-byte aligned");
  const int64_t n16 = (int64_t)(bytes / 16);
  const int blocks = (int)std::min<int64_t>((n16 + 255) / 256, (int64_t)num_sms());
  launch_kernel(copy_tables_kernel, blocks, 256, 0, stream, static_cast<const uint4*>(src),
                                                  static_cast<uint4*>(dst), n16);
  OES_CHECK_LAUNCH("copy_tables_kernel");
  return OES_OK;
}

}  // namespace

int64_t copy_run_items(int64_t bytes) {
  const int64_t item = (int64_t)kCopyThreads * kCopyUnroll * 16;
  return (bytes + item - 1) / item;
}

int launch_copy_runs(const void* src, void* dst, const CopyRun* runs, int nruns, int64_t src_off,
                     int64_t dst_off, int64_t bytes, int64_t nitems, cudaStream_t stream) {
  if (nitems <= 0) return OES_OK;
  if (const int rc = prefer_max_shared_carveout(reinterpret_cast<const void*>(copy_runs_kernel),
                                                "copy_runs_kernel: carveout"))
    return rc;
  const CopyRun one{src_off, dst_off, bytes, 0};
  launch_kernel(copy_runs_kernel, num_sms(), kCopyThreads, 0, stream, static_cast<const uint8_t*>(src),
                                                          static_cast<uint8_t*>(dst), runs, nruns,
                                                          one, nitems);
  OES_CHECK_LAUNCH("copy_runs_kernel");
  return OES_OK;
}

}  // namespace oes

using namespace oes;

// Frees whatever part of a cache handle exists (creation failures included).
static int release_cache(oes_slot_cache* c) {
  for (int q = 0; q < oes_slot_cache::kMaxQueries; ++q) {
    if (c->ensured[q]) cudaEventDestroy(c->ensured[q]);
    if (c->copied[2 * q]) cudaEventDestroy(c->copied[2 * q]);
    if (c->copied[2 * q + 1]) cudaEventDestroy(c->copied[2 * q + 1]);
  }
  if (c->join) cudaEventDestroy(c->join);
  if (c->fork) cudaEventDestroy(c->fork);
  if (c->prepared) cudaEventDestroy(c->prepared);
  if (c->gjoin) cudaEventDestroy(c->gjoin);
  if (c->routed) cudaEventDestroy(c->routed);
  if (c->flagged) cudaEventDestroy(c->flagged);
  if (c->side) cudaStreamDestroy(c->side);
  if (c->gemm) cudaStreamDestroy(c->gemm);
  cudaError_t e = c->block ? cudaFree(c->block) : cudaSuccess;
  delete c;
  if (e != cudaSuccess) return cuda_fail(e, "cudaFree(slot cache tables)");
  return OES_OK;
}

// LRFU scores 1.0 for occupied slots, 0 for empty ones; no pins.
static int reset_lrfu(oes_slot_cache* c, const int32_t* slot_key) {
  std::vector<uint64_t> crf(c->S);
  for (int s = 0; s < c->S; ++s) crf[s] = slot_key[s] >= 0 ? kCrfOne : 0;
  OES_TRY_CUDA(cudaMemcpy(c->crf, crf.data(), (size_t)c->S * 8, cudaMemcpyHostToDevice));
  OES_TRY_CUDA(cudaMemset(c->pin, 0, (size_t)c->S * 4));
  OES_TRY_CUDA(cudaMemset(c->ctr + 4, 0, 8));  // chunk tags start again at 1
  return OES_OK;
}

extern "C" int slot_cache_create(int S, int L, int E, oes_slot_cache** out) {
  OES_REQUIRE(out, "slot_cache_create: null out");
  OES_REQUIRE(S >= 1 && S <= OES_MAX_SLOTS, "slot_cache_create: S=%d out of [1, %d]", S,
              OES_MAX_SLOTS);
  OES_REQUIRE(E >= 1 && E <= OES_MAX_EXPERTS && L >= 1 && (int64_t)L * E < (1ll << 31),
              "slot_cache_create: bad L=%d E=%d", L, E);
  auto* c = new oes_slot_cache();
  c->S = S;
  c->L = L;
  c->E = E;
  cudaGetDevice(&c->device);
  const size_t LE = (size_t)L * E;
  const size_t bytes = (LE * 4 + (size_t)S * 4 + (size_t)S * 8 + 8 * 8 + LE * 8 + (size_t)S * 8 +
                        (size_t)S * 4 + 64 + 15) / 16 * 16;
  c->block_bytes = bytes;
  c->block = nullptr;
  cudaError_t e = cudaMalloc(&c->block, bytes);
  if (e == cudaSuccess) e = cudaMemset(c->block, 0, bytes);  // slack bytes included
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->gemm, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->join, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->prepared, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->gjoin, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->routed, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->flagged, cudaEventDisableTiming);
  for (int q = 0; q < oes_slot_cache::kMaxQueries && e == cudaSuccess; ++q) {
    e = cudaEventCreateWithFlags(&c->ensured[q], cudaEventDisableTiming);
    for (int p = 0; p < 2 && e == cudaSuccess; ++p)
      e = cudaEventCreateWithFlags(&c->copied[2 * q + p], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {
    release_cache(c);
    return cuda_fail(e, "slot_cache_create: tables, side stream or events");
  }
  uint8_t* p = static_cast<uint8_t*>(c->block);
  c->slot_ts = reinterpret_cast<int64_t*>(p);
  p += (size_t)S * 8;
  c->ctr = reinterpret_cast<int64_t*>(p);  // clock, hits, misses, evictions, chunk tag
  p += 8 * 8;
  c->decode_freq = reinterpret_cast<int64_t*>(p);
  p += LE * 8;
  c->crf = reinterpret_cast<uint64_t*>(p);
  p += (size_t)S * 8;
  c->map = reinterpret_cast<int32_t*>(p);
  p += LE * 4;
  c->slot_key = reinterpret_cast<int32_t*>(p);
  p += (size_t)S * 4;
  c->pin = reinterpret_cast<int32_t*>(p);
  c->policy = OES_POLICY_LRU;
  c->lrfu_k = 0;
  std::vector<int32_t> key(S, -1);
  std::vector<int64_t> ts(S, 0);
  int rc = slot_cache_load_state(c, key.data(), ts.data(), 0);
  if (rc != OES_OK) {
    release_cache(c);
    return rc;
  }
  *out = c;
  return OES_OK;
}

extern "C" int slot_cache_destroy(oes_slot_cache* c) {
  if (!c) return OES_OK;
  // the handle's own streams may still run kernels that read the tables
  if (c->side) cudaStreamSynchronize(c->side);
  if (c->gemm) cudaStreamSynchronize(c->gemm);
  return release_cache(c);
}

extern "C" int slot_cache_load_state(oes_slot_cache* c, const int32_t* slot_key,
                                     const int64_t* slot_ts, int64_t clock) {
  OES_REQUIRE(c && slot_key && slot_ts, "slot_cache_load_state: null pointer");
  OES_REQUIRE(clock >= 0 && clock < (1ll << 47), "slot_cache_load_state: bad clock %lld",
              (long long)clock);
  const int S = c->S;
  const int64_t LE = (int64_t)c->L * c->E;
  std::vector<int32_t> map(LE, -1);
  for (int s = 0; s < S; ++s) {
    const int32_t k = slot_key[s];
    OES_REQUIRE(k >= -1 && k < LE, "slot_cache_load_state: slot %d holds key %d out of range", s, k);
    if (k >= 0) {
      OES_REQUIRE(map[k] < 0, "slot_cache_load_state: key %d held by two slots", k);
      OES_REQUIRE(slot_ts[s] >= 1 && slot_ts[s] <= clock,
                  "slot_cache_load_state: slot %d timestamp %lld out of [1, clock]", s,
                  (long long)slot_ts[s]);
      map[k] = s;
    }
  }
  std::vector<int64_t> ts(S);
  for (int s = 0; s < S; ++s) ts[s] = slot_key[s] < 0 ? 0 : slot_ts[s];
  int64_t ctr[8] = {clock, 0, 0, 0, 0, 0, 0, 0};
  OES_TRY_CUDA(cudaMemcpy(c->map, map.data(), LE * 4, cudaMemcpyHostToDevice));
  OES_TRY_CUDA(cudaMemcpy(c->slot_key, slot_key, (size_t)S * 4, cudaMemcpyHostToDevice));
  OES_TRY_CUDA(cudaMemcpy(c->slot_ts, ts.data(), (size_t)S * 8, cudaMemcpyHostToDevice));
  OES_TRY_CUDA(cudaMemcpy(c->ctr, ctr, sizeof(ctr), cudaMemcpyHostToDevice));
  OES_TRY_CUDA(cudaMemset(c->decode_freq, 0, LE * 8));
  return reset_lrfu(c, slot_key);
}

extern "C" int slot_cache_reset(oes_slot_cache* c, oes_stream_t stream) {
  OES_REQUIRE(c, "slot_cache_reset: null cache");
  const int64_t LE = (int64_t)c->L * c->E;
  uint8_t* base = static_cast<uint8_t*>(c->block);
  uint8_t* map = reinterpret_cast<uint8_t*>(c->map);
  uint8_t* pin = reinterpret_cast<uint8_t*>(c->pin);
  // slot_ts, counters, decode_freq and LRFU scores precede the map; map and
  // slot_key are adjacent and become -1; the pins and the block's slack zero
  OES_TRY_CUDA(cudaMemsetAsync(base, 0, (size_t)(map - base), stream));
  OES_TRY_CUDA(cudaMemsetAsync(map, 0xff, (size_t)(LE + c->S) * 4, stream));
  OES_TRY_CUDA(cudaMemsetAsync(pin, 0, c->block_bytes - (size_t)(pin - base), stream));
  return OES_OK;
}

extern "C" int slot_cache_set_policy(oes_slot_cache* c, int policy, int lrfu_k) {
  OES_REQUIRE(c, "slot_cache_set_policy: null cache");
  OES_REQUIRE(policy == OES_POLICY_LRU || policy == OES_POLICY_LRFU,
              "slot_cache_set_policy: unknown policy %d", policy);
  OES_REQUIRE(lrfu_k >= 0 && lrfu_k <= OES_LRFU_MAX_K, "slot_cache_set_policy: k=%d out of [0, %d]",
              lrfu_k, OES_LRFU_MAX_K);
  OES_TRY_CUDA(cudaDeviceSynchronize());
  std::vector<int32_t> key(c->S);
  OES_TRY_CUDA(cudaMemcpy(key.data(), c->slot_key, (size_t)c->S * 4, cudaMemcpyDeviceToHost));
  c->policy = policy;
  c->lrfu_k = lrfu_k;
  return reset_lrfu(c, key.data());
}

extern "C" int slot_cache_read_lrfu(const oes_slot_cache* c, uint64_t* crf, int32_t* pin,
                                    oes_stream_t stream) {
  OES_REQUIRE(c, "slot_cache_read_lrfu: null cache");
  OES_TRY_CUDA(cudaStreamSynchronize(stream));
  if (crf) OES_TRY_CUDA(cudaMemcpy(crf, c->crf, (size_t)c->S * 8, cudaMemcpyDeviceToHost));
  if (pin) OES_TRY_CUDA(cudaMemcpy(pin, c->pin, (size_t)c->S * 4, cudaMemcpyDeviceToHost));
  return OES_OK;
}

extern "C" int slot_cache_read_state(const oes_slot_cache* c, int32_t* map, int32_t* slot_key,
                                     int64_t* slot_ts, int64_t* clock, int64_t* counters,
                                     int64_t* decode_freq, oes_stream_t stream) {
  OES_REQUIRE(c, "slot_cache_read_state: null cache");
  OES_TRY_CUDA(cudaStreamSynchronize(stream));
  const size_t LE = (size_t)c->L * c->E;
  if (map) OES_TRY_CUDA(cudaMemcpy(map, c->map, LE * 4, cudaMemcpyDeviceToHost));
  if (slot_key)
    OES_TRY_CUDA(cudaMemcpy(slot_key, c->slot_key, (size_t)c->S * 4, cudaMemcpyDeviceToHost));
  if (slot_ts)
    OES_TRY_CUDA(cudaMemcpy(slot_ts, c->slot_ts, (size_t)c->S * 8, cudaMemcpyDeviceToHost));
  int64_t ctr[4];
  OES_TRY_CUDA(cudaMemcpy(ctr, c->ctr, sizeof(ctr), cudaMemcpyDeviceToHost));
  if (clock) *clock = ctr[0];
  if (counters) {
    counters[0] = ctr[1];
    counters[1] = ctr[2];
    counters[2] = ctr[3];
  }
  if (decode_freq)
    OES_TRY_CUDA(cudaMemcpy(decode_freq, c->decode_freq, LE * 8, cudaMemcpyDeviceToHost));
  return OES_OK;
}

extern "C" size_t slot_cache_state_bytes(const oes_slot_cache* c) { return c ? c->block_bytes : 0; }

extern "C" int slot_cache_snapshot(const oes_slot_cache* c, void* dst, oes_stream_t stream) {
  OES_REQUIRE(c && dst, "slot_cache_snapshot: null pointer");
  return copy_tables(c->block, dst, c->block_bytes, stream);
}

extern "C" int slot_cache_restore(oes_slot_cache* c, const void* src, oes_stream_t stream) {
  OES_REQUIRE(c && src, "slot_cache_restore: null pointer");
  return copy_tables(src, c->block, c->block_bytes, stream);
}

extern "C" int slot_cache_layer_map(const oes_slot_cache* c, int layer, const int32_t** e2s) {
  OES_REQUIRE(c && e2s, "slot_cache_layer_map: null pointer");
  OES_REQUIRE(layer >= 0 && layer < c->L, "slot_cache_layer_map: layer %d out of [0, %d)", layer,
              c->L);
  *e2s = c->map + (size_t)layer * c->E;
  return OES_OK;
}

extern "C" int slot_cache_ensure_tagged(oes_slot_cache* c, int layer, const int32_t* experts,
                                        int n, int record_stats, int32_t tag, int32_t* miss,
                                        int32_t* n_miss, int32_t* status, oes_stream_t stream) {
  OES_REQUIRE(c && miss && n_miss && (n == 0 || experts), "slot_cache_ensure: null pointer");
  OES_REQUIRE(layer >= 0 && layer < c->L, "slot_cache_ensure: layer %d out of [0, %d)", layer, c->L);
  OES_REQUIRE(tag >= 0 || tag == OES_TAG_NEW_CHUNK || tag == OES_TAG_SAME_CHUNK,
              "slot_cache_ensure_tagged: tag %d is neither >= 0 nor a chunk-tag code", tag);
  OES_REQUIRE(n >= 0 && n <= OES_QUERY_MAX, "slot_cache_ensure: n=%d out of [0, %d]", n,
              OES_QUERY_MAX);
  int spad = 2;
  while (spad < c->S) spad <<= 1;
  const size_t smem = (size_t)spad * 8;
  int rc;
  if (smem > 48 * 1024 &&
      (rc = set_max_dynamic_smem(reinterpret_cast<const void*>(ensure_kernel), smem,
                                 "ensure_kernel: shared memory limit")))
    return rc;
  // the largest shared carveout, as for the copies (an ensure may run beside
  // the copies and the GEMM)
  if ((rc = prefer_max_shared_carveout(reinterpret_cast<const void*>(ensure_kernel),
                                       "ensure_kernel: carveout")))
    return rc;
  launch_kernel(ensure_kernel, 1, kEnsureThreads, smem, stream, view_of(c), layer, experts, n, record_stats,
                                                     tag, spad, miss, n_miss, status);
  OES_CHECK_LAUNCH("ensure_kernel");
  return OES_OK;
}

extern "C" int slot_cache_ensure(oes_slot_cache* c, int layer, const int32_t* experts, int n,
                                 int record_stats, int32_t* miss, int32_t* n_miss, int32_t* status,
                                 oes_stream_t stream) {
  return slot_cache_ensure_tagged(c, layer, experts, n, record_stats, 0, miss, n_miss, status,
                                  stream);
}

extern "C" int oes_expert_source_create(const void* const* layer_base, int L, int E,
                                        int64_t row_bytes, oes_expert_source** out) {
  OES_REQUIRE(out && layer_base, "oes_expert_source_create: null pointer");
  OES_REQUIRE(L >= 1 && E >= 1 && (int64_t)L * E < (1ll << 31), "oes_expert_source_create: bad L/E");
  OES_REQUIRE(row_bytes > 0 && row_bytes % 16 == 0,
              "oes_expert_source_create: row_bytes %lld is not a positive multiple of 16",
              (long long)row_bytes);
  for (int l = 0; l < L; ++l)
    OES_REQUIRE(layer_base[l] && ((uintptr_t)layer_base[l] & 15) == 0,
                "oes_expert_source_create: layer %d base is null or not 16-byte aligned", l);
  auto* s = new oes_expert_source();
  s->L = L;
  s->E = E;
  s->row_bytes = row_bytes;
  s->host_bases.assign(layer_base, layer_base + L);
  s->dev_bases = nullptr;
  cudaError_t e = cudaMalloc(&s->dev_bases, sizeof(void*) * L);
  if (e == cudaSuccess)
    e = cudaMemcpy(s->dev_bases, s->host_bases.data(), sizeof(void*) * L, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(s->dev_bases);
    delete s;
    return cuda_fail(e, "oes_expert_source_create");
  }
  *out = s;
  return OES_OK;
}

extern "C" int oes_expert_source_destroy(oes_expert_source* s) {
  if (!s) return OES_OK;
  cudaError_t e = cudaFree(s->dev_bases);
  delete s;
  if (e != cudaSuccess) return cuda_fail(e, "cudaFree(source bases)");
  return OES_OK;
}

namespace oes {
int copy_misses_part(const oes_expert_source* src, void* pool, int S, const int32_t* miss,
                     const int32_t* n_miss, int max_misses, int part, int32_t* status,
                     cudaStream_t stream) {
  OES_REQUIRE(src && pool && miss && n_miss, "slot_cache_copy_misses: null pointer");
  OES_REQUIRE(S >= 1 && max_misses >= 0 && max_misses <= OES_QUERY_MAX,
              "slot_cache_copy_misses: bad S=%d max_misses=%d", S, max_misses);
  OES_REQUIRE(((uintptr_t)pool & 15) == 0, "slot_cache_copy_misses: pool not 16-byte aligned");
  if (max_misses == 0) return OES_OK;
  // the copies run beside kernels that need most of an SM's shared memory;
  // an SM changes its L1 / shared split only when idle, so the copy kernel
  // asks for the largest shared carveout and never shrinks it
  if (const int rc = prefer_max_shared_carveout(reinterpret_cast<const void*>(copy_misses_kernel),
                                                "copy_misses_kernel: carveout"))
    return rc;
  const int grid = num_sms();
  launch_kernel(copy_misses_kernel, grid, kCopyThreads, 0, stream, src->dev_bases, src->L, src->E,
                src->row_bytes, static_cast<uint8_t*>(pool), S, miss, n_miss, max_misses, part,
                status);
  OES_CHECK_LAUNCH("copy_misses_kernel");
  return OES_OK;
}
}  // namespace oes

extern "C" int slot_cache_copy_misses(const oes_expert_source* src, void* pool, int S,
                                      const int32_t* miss, const int32_t* n_miss, int max_misses,
                                      int32_t* status, oes_stream_t stream) {
  return copy_misses_part(src, pool, S, miss, n_miss, max_misses, -1, status, stream);
}

extern "C" int oes_copy_layer(const oes_expert_source* src, int layer, void* dst,
                              oes_stream_t stream) {
  OES_REQUIRE(src && dst, "oes_copy_layer: null pointer");
  OES_REQUIRE(layer >= 0 && layer < src->L, "oes_copy_layer: layer %d out of range", layer);
  OES_REQUIRE(((uintptr_t)dst & 15) == 0, "oes_copy_layer: dst not 16-byte aligned");
  const int64_t bytes = (int64_t)src->E * src->row_bytes;
  return launch_copy_runs(src->host_bases[layer], dst, nullptr, 0, 0, 0, bytes,
                          copy_run_items(bytes), stream);
}
