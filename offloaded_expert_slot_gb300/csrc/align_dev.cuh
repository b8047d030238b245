// Device code of the single-CTA align (moe_align_block_size of up to
// kSmallR routes), shared by its kernel and the fused decode step
// (FreeToken PR #676, Solution and Tests: each route placed exactly once, in
// a block of its own expert).
#pragma once
#include "common.cuh"

namespace oes {

// The whole align for up to kSmallR routes in one CTA of 1024 threads (a
// decode step's routes: one launch instead of three).  Same output, bit for
// bit: histogram, the padded exclusive scan over experts, each route placed
// at its expert's offset plus the number of earlier routes of that expert
// (counted directly: at most kSmallR^2 / 1024 comparisons a thread), and the
// padding and block experts of every block up to the capacity.
constexpr int kSmallR = 1024;

// sm: shared memory of 2E + max(R, 1) int32.  Plain loads of ids: the fused
// decode step writes them in the same kernel.
__device__ __forceinline__ void align_small_cta(const int32_t* ids, int R, int E, int B, int64_t cap,
                                                int ignore_invalid, int32_t* __restrict__ sorted_ids,
                                                int32_t* __restrict__ block_expert,
                                                int32_t* __restrict__ n_post_pad,
                                                int32_t* __restrict__ status, int32_t* __restrict__ zero,
                                                int nzero, int32_t* sm) {
  for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
  int32_t* cnt = sm;           // [E]
  int32_t* off = sm + E;       // [E]
  int32_t* sid = sm + 2 * E;   // [R] expert of each route, -1 if invalid
  __shared__ int warp_tot[32];
  __shared__ int s_total;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, w = tid >> 5;
  for (int e = tid; e < E; e += nt) cnt[e] = 0;
  bool bad = false;
  for (int r = tid; r < R; r += nt) {
    const int v = ids[r];
    const bool ok = v >= 0 && v < E;
    sid[r] = ok ? v : -1;
    bad |= !ok;
  }
  if (bad && !ignore_invalid) set_status(status, OES_DEV_BAD_ID);
  __syncthreads();
  for (int r = tid; r < R; r += nt)
    if (sid[r] >= 0) atomicAdd(&cnt[sid[r]], 1);
  __syncthreads();
  // padded sizes -> exclusive offsets over experts
  const int per = (E + nt - 1) / nt;
  const int b0 = min(E, tid * per), b1 = min(E, b0 + per);
  int sum = 0;
  for (int e = b0; e < b1; ++e) sum += (cnt[e] + B - 1) / B * B;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int nw = nt >> 5;
    int t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += x;
    }
    if (lane < nw) warp_tot[lane] = t;
    if (lane == nw - 1) s_total = t;
  }
  __syncthreads();
  int run = incl - sum + (w ? warp_tot[w - 1] : 0);
  for (int e = b0; e < b1; ++e) {
    off[e] = run;
    run += (cnt[e] + B - 1) / B * B;
  }
  __syncthreads();
  const int total = s_total;
  if (tid == 0) *n_post_pad = total;
  // routes, stable within each expert
  for (int r = tid; r < R; r += nt) {
    const int v = sid[r];
    if (v < 0) continue;
    int rank = 0;
    for (int q = 0; q < r; ++q) rank += sid[q] == v ? 1 : 0;
    sorted_ids[off[v] + rank] = r;
  }
  // padding and block experts
  const int nblk = total / B;
  for (int64_t b = tid; b < cap / B; b += nt) {
    int e = -1;
    int64_t first_pad = b * B;
    if (b < nblk) {
      int lo = 0, hi = E - 1;  // largest e with off[e] <= b*B
      const int x = (int)(b * B);
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= x) lo = mid;
        else hi = mid - 1;
      }
      e = lo;
      first_pad = (int64_t)off[e] + cnt[e];
    }
    block_expert[b] = e;
    for (int i = 0; i < B; ++i) {
      const int64_t p = b * B + i;
      if (p >= first_pad) sorted_ids[p] = R;
    }
  }
}

}  // namespace oes
