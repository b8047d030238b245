// Library-private definitions shared by the .cu files of liboes.
#pragma once

#include <stdint.h>

#include <vector>

#include <cuda_runtime.h>

#include "oes.h"

struct oes_slot_cache {
  int S, L, E, device;
  void* block;           // one allocation for every table
  size_t block_bytes;
  int32_t* map;          // [L*E] slot of each key, -1 if absent
  int32_t* slot_key;     // [S] key held by each slot, -1 if empty
  int64_t* slot_ts;      // [S] timestamp of the last query that touched the slot, 0 if empty
  int64_t* ctr;          // [4] clock, hits, misses, evictions
  int64_t* decode_freq;  // [L*E]
  uint64_t* crf;         // [S] LRFU score of each slot, Q32.32
  int32_t* pin;          // [S] LRFU pin tag of each slot, 0 = none
  int policy, lrfu_k;    // OES_POLICY_*, LRFU decay shift
  // streams and events of moe_layer_forward_slots: the later queries'
  // ensures, the group flags and the GEMM over the hits run on `side`; the
  // align, the GEMMs' x and the GEMM over each part of each query's copied
  // experts on `gemm`; the misses are copied on the caller's stream.
  // routed marks the routing, ensured[q] query q's ensure, flagged the
  // group flags, copied[2q + p] the copies of part p of query q's misses,
  // prepared the align and x, join / gjoin the ends of side / gemm
  static constexpr int kMaxQueries = OES_MAX_EXPERTS / OES_QUERY_MAX;
  cudaStream_t side = nullptr, gemm = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, prepared = nullptr, gjoin = nullptr;
  cudaEvent_t routed = nullptr, flagged = nullptr;
  cudaEvent_t ensured[kMaxQueries] = {}, copied[2 * kMaxQueries] = {};
};

struct oes_expert_source {
  int L, E;
  int64_t row_bytes;
  std::vector<const void*> host_bases;  // [L] mapped addresses
  const uint8_t** dev_bases;            // device copy of host_bases
};

namespace oes {
int tile_plan(int R, int E);
// moe_align_block_size, which also zeroes nzero int32 words at `zero` (device)
// in one of its kernels: a composite call clears the GEMM's K-split counters
// there instead of in a memset of its own.
int align_run(const int32_t* ids, int R, int E, int B, int ignore_invalid, int32_t* sorted_ids,
              int32_t* block_expert, int32_t* n_post_pad, int32_t* status, void* workspace,
              size_t workspace_bytes, int32_t* zero, int nzero, cudaStream_t stream);

// The slot path copies the n misses of a query of more than kSplitIds ids in
// two parts, so that the GEMM over the first part's experts runs while the
// last part is still being copied: part 0 = misses [0, miss_split(n)),
// part 1 = the last min(n / 2, 16).  A smaller query's GEMM is one wave of
// CTAs either way, and its misses go in one part.
constexpr int kSplitIds = 32;
__host__ __device__ inline int miss_split(int n) { return n - (n / 2 < 16 ? n / 2 : 16); }
// Expert groups of the slot path's filtered GEMM launches: 0 not in the
// chunk, kGroupHit a hit in its own query, kGroupMiss0 + 2q + p missed in
// part p of query q's misses.
constexpr int kGroupHit = 1, kGroupMiss0 = 2;
constexpr int kGroups = kGroupMiss0 + 2 * (OES_MAX_EXPERTS / OES_QUERY_MAX);
// slot_cache_copy_misses for part 0 or 1 of the query's misses (-1: all).
int copy_misses_part(const oes_expert_source* src, void* pool, int S, const int32_t* miss,
                     const int32_t* n_miss, int max_misses, int part, int32_t* status,
                     cudaStream_t stream);

// A contiguous run of bytes from a host-mapped source to device memory;
// item0 = the run's first 4 KB item in its copy launch.
struct CopyRun {
  int64_t src_off, dst_off, bytes, item0;
};
int64_t copy_run_items(int64_t bytes);
// Copies the runs (device [nruns]) or, when runs is null, the one run
// (src_off, dst_off, bytes); nitems = the launch's 4 KB items in all.
int launch_copy_runs(const void* src, void* dst, const CopyRun* runs, int nruns, int64_t src_off,
                     int64_t dst_off, int64_t bytes, int64_t nitems, cudaStream_t stream);
}  // namespace oes
