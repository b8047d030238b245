// Device code of the routing steps, shared by their own kernels and by the
// fused decode step (top-k of a token by one warp, distinct experts by one
// CTA).  FreeToken PR #676, Solution: the chunk's distinct experts are what
// the cache is asked for.
#pragma once
#include "common.cuh"

namespace oes {

__device__ __forceinline__ float load_logit(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_logit(const uint16_t* p) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(p)) << 16);  // bf16 -> fp32, exact
}

// Order key of a routing logit: a larger logit has a larger key, and the
// key order is the order the router ranks by.  NaN ranks as -inf (fmaxf
// returns the number when one operand is NaN) and -0 as +0 (x + 0 is +0 for
// x = -0), so that equal logits get equal keys; key 0 marks an entry that is
// not an expert or is already taken (every logit's key is at least that of
// -inf, 0x007FFFFF).
__device__ __forceinline__ uint32_t logit_key(float v) {
  const uint32_t u = __float_as_uint(fmaxf(v, -INFINITY) + 0.0f);
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// The three best entries (key, position j) of a lane's EPL keys, skipping the
// positions set in `taken`; ties go to the lower j (strict comparisons in
// ascending j).  Position EPL and key 0 mean none.
template <int EPL>
__device__ __forceinline__ void lane_top3(const uint32_t (&key)[EPL], uint32_t taken, uint32_t (&kb)[3],
                                          int (&jb)[3]) {
  kb[0] = kb[1] = kb[2] = 0u;
  jb[0] = jb[1] = jb[2] = EPL;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const uint32_t kj = (j < 32 && ((taken >> (j & 31)) & 1u)) ? 0u : key[j];
    if (kj > kb[0]) {
      kb[2] = kb[1];
      jb[2] = jb[1];
      kb[1] = kb[0];
      jb[1] = jb[0];
      kb[0] = kj;
      jb[0] = j;
    } else if (kj > kb[1]) {
      kb[2] = kb[1];
      jb[2] = jb[1];
      kb[1] = kj;
      jb[1] = j;
    } else if (kj > kb[2]) {
      kb[2] = kj;
      jb[2] = j;
    }
  }
}

// Lane r < k holds the key and expert id of rank r: writes the ids and the
// softmax over the k selected logits (a butterfly sum over the lanes in rank
// order, so the weights depend only on the selected logits and their ranks).
__device__ __forceinline__ void topk_write(uint32_t my_k, uint32_t my_e, int k, int lane,
                                           int32_t* __restrict__ ids_t, float* __restrict__ w_t) {
  const float my_v = key_logit(my_k);
  const float top = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - top) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    ids_t[lane] = (int32_t)my_e;
    w_t[lane] = ex / sum;
  }
}

// One token's top-k by one warp, in rounds.  Lane l holds the keys of its
// experts (topk_row: l, l + 32, ...; logits widened to fp32, bf16 exactly)
// and its three best.  Each of the k
// rounds takes the warp's largest key (one redux.sync), then the lowest
// expert id holding it (another): larger logit first, ties to the lower id.
// Only the winning lane moves on to its next entry: its next best, or, once
// its three are used, a rescan of its keys without the taken ones (a bit
// mask of taken positions up to 32 keys a lane; past that the key is
// cleared).  Lane r keeps round r's winner; the weights are a softmax over
// the k selected logits.
// Expert id of a lane's j-th key when each lane holds V consecutive experts
// of every 32 V: V lane + 32 V (j / V) + j % V (lane + 32 j for V = 1),
// increasing in j, so the lower j of a lane is the lower id.
template <int V>
__device__ __forceinline__ uint32_t lane_expert(int lane, int j) {
  return (uint32_t)(V * lane + 32 * V * (j / V) + j % V);
}

template <int EPL, int V>
__device__ __forceinline__ void topk_rounds(uint32_t (&key)[EPL], int k, int lane, int32_t* __restrict__ ids_t,
                                            float* __restrict__ w_t) {
  // the lane's three best untaken keys; `left` of them after the first
  uint32_t kb[3];
  int jb[3];
  lane_top3<EPL>(key, 0u, kb, jb);
  int left = 2;
  uint32_t taken = 0u;
  uint32_t my_k = 0u, my_e = 0u;
  for (int r = 0; r < k; ++r) {
    const uint32_t g = __reduce_max_sync(0xffffffffu, kb[0]);
    const uint32_t cand = (kb[0] == g) ? lane_expert<V>(lane, jb[0]) : 0xffffffffu;
    const uint32_t we = __reduce_min_sync(0xffffffffu, cand);
    if (lane == r) {
      my_k = g;
      my_e = we;
    }
    if (lane == (int)((we / V) & 31u)) {  // the lane holding expert we
      if (EPL <= 32) {
        taken |= 1u << (jb[0] & 31);
      } else {
        // wider rows (more than 1024 experts) clear the taken key in place
#pragma unroll
        for (int j = 0; j < EPL; ++j)
          if (j == jb[0]) key[j] = 0u;
      }
      if (left > 0) {
        kb[0] = kb[1];
        jb[0] = jb[1];
        kb[1] = kb[2];
        jb[1] = jb[2];
        --left;
      } else {
        lane_top3<EPL>(key, taken, kb, jb);
        left = 2;
      }
    }
  }
  topk_write(my_k, my_e, k, lane, ids_t, w_t);
}

template <int EPL, typename LT>
__device__ __forceinline__ void topk_row(const LT* __restrict__ row, int E, int k, int lane,
                                         int32_t* __restrict__ ids_t, float* __restrict__ w_t) {
  uint32_t key[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = lane + 32 * j;
    key[j] = (e < E) ? logit_key(load_logit(row + e)) : 0u;
  }
  topk_rounds<EPL, 1>(key, k, lane, ids_t, w_t);
}

// V consecutive logits from p, widened to fp32 (bf16 exactly); V > 1 wants p
// 16-byte aligned.
template <int V>
__device__ __forceinline__ void load_logits(const float* p, float* o) {
  if constexpr (V == 4) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(p));
    o[0] = f.x;
    o[1] = f.y;
    o[2] = f.z;
    o[3] = f.w;
  } else {
    static_assert(V == 1, "fp32 logits: 1 or 4 a load");
    o[0] = __ldg(p);
  }
}
template <int V>
__device__ __forceinline__ void load_logits(const uint16_t* p, float* o) {
  if constexpr (V == 8) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
    static_assert(V == 1, "bf16 logits: 1 or 8 a load");
    o[0] = load_logit(p);
  }
}

// The same top-k as topk_row, by a threshold filter.  Lane l holds experts
// V l + 32 V q + i (q < Q, i < V).  Let tau be the k-th largest of the 32
// lane maxima (a bitonic sort of them): at least k logits are >= tau (those
// maxima), so every logit of the top k is >= tau, and for random rows only a
// few more are.  The candidates (logit >= tau) go to `cand` (this warp's own
// 33 entries: 32 candidates, then the count) at positions from a shared
// counter, in any order; each ranks itself against the others by (key, lower
// id) and rank r goes to lane r.  A row whose tau is -inf (fewer than k lanes
// with a number above -inf: NaN and missing experts rank lowest) or that has
// more than 32 candidates (many equal logits) is ranked in rounds over the
// same keys.  Both give the same ids and, through topk_write, the same
// weights bit for bit.
template <int V, int Q, typename LT>
__device__ __forceinline__ void topk_row_filtered(const LT* __restrict__ row, int E, int k, int lane,
                                                  int32_t* __restrict__ ids_t, float* __restrict__ w_t,
                                                  uint2* cand) {
  constexpr int EPL = V * Q;
  int* count = reinterpret_cast<int*>(cand + 32);
  float v[EPL];
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const int e0 = V * lane + 32 * V * q;
    if (e0 + V <= E) {
      load_logits<V>(row + e0, v + V * q);
    } else {
#pragma unroll
      for (int i = 0; i < V; ++i) v[V * q + i] = __int_as_float(0x7fffffff);  // NaN: no expert
    }
  }
  float m = -INFINITY;  // fmaxf skips NaN
#pragma unroll
  for (int j = 0; j < EPL; ++j) m = fmaxf(m, v[j]);
  // tau: the k-th largest lane maximum, from a bitonic sort of the 32
  // maxima into descending order (lane i the i-th largest)
  float srt = m;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int d = size >> 1; d > 0; d >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, srt, d);
      srt = (((lane & d) == 0) == ((lane & size) == 0)) ? fmaxf(srt, o) : fminf(srt, o);
    }
  const float tau = __shfl_sync(0xffffffffu, srt, k - 1);
  bool rounds = tau == -INFINITY;
  int N = 0;
  if (!rounds) {
    __syncwarp();  // the previous row's reads of cand are done
    if (lane == 0) *count = 0;
    __syncwarp();
#pragma unroll
    for (int q = 0; q < Q; ++q)
#pragma unroll
      for (int i = 0; i < V; ++i)
        if (v[V * q + i] >= tau) {
          const int p = atomicAdd(count, 1);
          if (p < 32) cand[p] = make_uint2(__float_as_uint(v[V * q + i]), V * lane + 32 * V * q + i);
        }
    __syncwarp();
    N = *count;
    rounds = N > 32;
  }
  if (rounds) {
    uint32_t key[EPL];
#pragma unroll
    for (int q = 0; q < Q; ++q)
#pragma unroll
      for (int i = 0; i < V; ++i)
        key[V * q + i] = (V * lane + 32 * V * q + V <= E) ? logit_key(v[V * q + i]) : 0u;
    topk_rounds<EPL, V>(key, k, lane, ids_t, w_t);
    return;
  }
  uint32_t ck = 0u, ce = 0u;
  uint64_t pk = 0u;
  if (lane < N) {
    const uint2 c = cand[lane];
    ck = logit_key(__uint_as_float(c.x));
    ce = c.y;
    pk = ((uint64_t)ck << 32) | (uint32_t)~ce;  // larger key first, then the lower id
  }
  int r = 0;
  for (int c = 0; c < N; ++c) r += (__shfl_sync(0xffffffffu, pk, c) > pk);
  __syncwarp();
  if (lane < N && r < k) cand[r] = make_uint2(ck, ce);
  __syncwarp();
  uint32_t my_k = 0u, my_e = 0u;
  if (lane < k) {
    const uint2 c = cand[lane];
    my_k = c.x;
    my_e = c.y;
  }
  topk_write(my_k, my_e, k, lane, ids_t, w_t);
}

// The distinct experts of R routes by one CTA: presence flags over the E
// experts in shared memory (flag: E bytes), then a block-wide exclusive scan
// turns flags into output positions.  Plain loads of ids: the fused decode
// step writes them in the same kernel.
__device__ __forceinline__ void distinct_cta(const int32_t* ids, int R, int E,
                                             int32_t* __restrict__ distinct,
                                             int32_t* __restrict__ d_count, uint8_t* flag) {
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int i = tid; i < E; i += nt) flag[i] = 0;
  __syncthreads();
  for (int r = tid; r < R; r += nt) {
    const int v = ids[r];
    if (v >= 0 && v < E) flag[v] = 1;
  }
  __syncthreads();
  const int per = (E + nt - 1) / nt;
  const int b0 = min(E, tid * per), b1 = min(E, b0 + per);
  int cnt = 0;
  for (int i = b0; i < b1; ++i) cnt += flag[i];
  const int lane = tid & 31, w = tid >> 5;
  int incl = cnt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int nw = nt >> 5;
    int s = (lane < nw) ? warp_tot[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += o;
    }
    if (lane < nw) warp_tot[lane] = s;  // inclusive per warp
  }
  __syncthreads();
  int pos = incl - cnt + (w ? warp_tot[w - 1] : 0);
  for (int i = b0; i < b1; ++i)
    if (flag[i]) distinct[pos++] = i;
  const int D = warp_tot[(nt >> 5) - 1];
  const int Lq = min(R, E);
  for (int i = D + tid; i < Lq; i += nt) distinct[i] = -1;
  if (tid == 0) *d_count = D;
}

}  // namespace oes
