// Device code of an ensure query (the LRU / LRFU slot cache's lookup, victim
// selection and table update), shared by the ensure kernel and the fused
// decode step.  FreeToken PR #676, Solution: the distinct experts reach
// lru_ensure in queries of at most 128; the author's reply on that page: LRU.
#pragma once
#include "common.cuh"
#include "internal.h"

namespace oes {

struct CacheView {
  int S, L, E;
  int32_t* map;
  int32_t* slot_key;
  int64_t* slot_ts;
  int64_t* ctr;
  int64_t* decode_freq;
  uint64_t* crf;
  int32_t* pin;
  int policy, lrfu_k;
};

inline CacheView view_of(oes_slot_cache* c) {
  return CacheView{c->S,   c->L,      c->E,           c->map, c->slot_key, c->slot_ts,
                   c->ctr, c->decode_freq, c->crf, c->pin,   c->policy,   c->lrfu_k};
}

constexpr uint64_t kCrfOne = 1ull << 32;           // LRFU score 1.0 (Q32.32)
constexpr uint64_t kCrfSat = (1ull << 51) - 1;     // saturation; leaves 13 bits for the slot

constexpr int kEnsureThreads = 1024;

// One ensure query by one CTA of kEnsureThreads threads; skey: shared
// memory of spad 64-bit words.  Victims: the nmiss smallest 64-bit keys of
// the non-hit slots, in ascending order, found by a radix select (no full
// sort).  LRU: key = (timestamp << 16 | slot); empty slots have timestamp 0
// and so come first, in slot order.  LRFU (Lee et al., IEEE Trans. Computers 2001, with
// F(x) = (1 - 2^-k)^x): every slot's score decays once (crf -= crf >> k),
// then key = (score << 13 | slot) over the slots that are neither hit nor
// pinned to this query's tag, empty slots scoring 0; hits gain 1.0, fills
// start at 1.0, and a nonzero tag pins every touched slot (gdevenyi's review
// comment on FreeToken PR #676: a scored policy must pin a chunk's earlier
// queries against its later ones).
__device__ __forceinline__ void ensure_query(CacheView c, int layer, const int32_t* __restrict__ experts,
                                             int n, int record_stats, int tag,
                                             int32_t* __restrict__ miss, int32_t* __restrict__ n_miss,
                                             int32_t* __restrict__ status, uint64_t* skey) {
  __shared__ int32_t qkey[OES_QUERY_MAX];
  __shared__ int32_t qslot[OES_QUERY_MAX];
  __shared__ int32_t qrank[OES_QUERY_MAX];
  __shared__ int32_t wvalid[4], wmiss[4];
  __shared__ uint32_t hitmask[OES_MAX_SLOTS / 32];
  __shared__ int32_t s_bad, s_nvalid, s_nmiss, s_nhit, s_evict, s_navail;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int LE = c.L * c.E;

  const bool lrfu = c.policy == OES_POLICY_LRFU;
  __shared__ int32_t s_tag;
  if (tid == 0) {
    s_bad = 0;
    s_evict = 0;
    s_navail = 0;
    // OES_TAG_NEW_CHUNK takes the next chunk tag from the tables (so that a
    // replayed graph gets a fresh one every time), OES_TAG_SAME_CHUNK the
    // current one; any other value is the tag itself
    int64_t t = tag;
    if (tag == OES_TAG_NEW_CHUNK) {
      t = c.ctr[4] >= INT32_MAX ? 1 : c.ctr[4] + 1;
      c.ctr[4] = t;
    } else if (tag == OES_TAG_SAME_CHUNK) {
      t = c.ctr[4];
    }
    s_tag = static_cast<int32_t>(t);
  }
  for (int i = tid; i < (c.S + 31) / 32; i += blockDim.x) hitmask[i] = 0;
  __syncthreads();
  const int use_tag = lrfu ? s_tag : 0;

  // 1. compact the valid ids of the query into keys
  int key = -1;
  bool valid = false;
  if (tid < OES_QUERY_MAX) {
    const int e = (tid < n) ? experts[tid] : -1;
    if (e != -1) {
      if (e < 0 || e >= c.E) {
        s_bad = 1;
      } else {
        valid = true;
        key = layer * c.E + e;
      }
    }
    const unsigned b = __ballot_sync(0xffffffffu, valid);
    if (lane == 0) wvalid[w] = __popc(b);
  }
  __syncthreads();
  if (tid < OES_QUERY_MAX) {
    const unsigned b = __ballot_sync(0xffffffffu, valid);
    int off = 0;
    for (int i = 0; i < w; ++i) off += wvalid[i];
    if (valid) qkey[off + __popc(b & ((1u << lane) - 1u))] = key;
  }
  if (tid == 0) s_nvalid = wvalid[0] + wvalid[1] + wvalid[2] + wvalid[3];
  __syncthreads();
  const int nvalid = s_nvalid;
  if (tid + 1 < nvalid && qkey[tid] >= qkey[tid + 1]) s_bad = 1;
  __syncthreads();
  if (s_bad || nvalid == 0) {
    if (tid == 0) {
      if (s_bad) set_status(status, OES_DEV_BAD_ID);
      *n_miss = 0;
    }
    return;
  }

  // 2. look the keys up; rank the misses in key order; mark hit slots
  bool is_miss = false;
  if (tid < OES_QUERY_MAX) {
    int slot = -1;
    if (tid < nvalid) {
      slot = c.map[qkey[tid]];
      if (slot >= c.S) {  // a corrupt table entry: treat as a miss and report
        set_status(status, OES_DEV_BAD_ID);
        slot = -1;
      }
      qslot[tid] = slot;
      if (slot >= 0) atomicOr(&hitmask[slot >> 5], 1u << (slot & 31));
      is_miss = slot < 0;
    }
    const unsigned b = __ballot_sync(0xffffffffu, is_miss);
    if (lane == 0) wmiss[w] = __popc(b);
  }
  __syncthreads();
  if (tid < OES_QUERY_MAX) {
    const unsigned b = __ballot_sync(0xffffffffu, is_miss);
    int off = 0;
    for (int i = 0; i < w; ++i) off += wmiss[i];
    qrank[tid] = is_miss ? off + __popc(b & ((1u << lane) - 1u)) : -1;
  }
  if (tid == 0) {
    s_nmiss = wmiss[0] + wmiss[1] + wmiss[2] + wmiss[3];
    s_nhit = nvalid - s_nmiss;
  }
  __syncthreads();
  const int nmiss = s_nmiss, nhit = s_nhit;
  const int slot_bits = lrfu ? 13 : 16;

  // 3. when there are misses: key the evictable slots (LRU: timestamp, LRFU:
  // decayed score; empty slots 0; every key unique by its slot bits) and
  // select the nmiss smallest keys, ascending, into vic[]: a radix select
  // finds the nmiss-th smallest key 8 bits at a time from the top
  // significant digit, then the keys at or below it are ranked by counting
  __shared__ uint64_t vic[OES_QUERY_MAX];
  __shared__ uint64_t vsel[OES_QUERY_MAX];
  __shared__ int hist[256];
  __shared__ uint32_t s_orw[2][32];
  __shared__ uint64_t s_prefix;
  __shared__ int s_need, s_nsel, s_hb;
  if (nmiss > 0) {
    uint64_t orv = 0;
    int navail = 0;
    for (int base = 0; base < c.S; base += blockDim.x) {
      const int s = base + tid;
      uint64_t k = ~0ull;
      if (s < c.S && !(hitmask[s >> 5] & (1u << (s & 31))) && !(use_tag && c.pin[s] == use_tag)) {
        uint64_t v;
        if (c.slot_key[s] < 0) {
          v = 0;
        } else if (lrfu) {
          const uint64_t crf = c.crf[s];
          v = min(c.lrfu_k ? crf - (crf >> c.lrfu_k) : crf, kCrfSat);
        } else {
          v = static_cast<uint64_t>(c.slot_ts[s]);
        }
        k = (v << slot_bits) | static_cast<uint64_t>(s);
        orv |= k;
      }
      if (s < c.S) skey[s] = k;
      navail += __popc(__ballot_sync(0xffffffffu, k != ~0ull));
    }
    const uint32_t olo = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(orv));
    const uint32_t ohi = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(orv >> 32));
    if (lane == 0) {
      atomicAdd(&s_navail, navail);
      s_orw[0][w] = olo;
      s_orw[1][w] = ohi;
    }
    __syncthreads();
    if (nmiss > s_navail) {
      if (tid == 0) {
        set_status(status, OES_DEV_CAPACITY);
        *n_miss = 0;
      }
      return;
    }
    if (tid == 0) {
      uint64_t o = 0;
      for (int i = 0; i < (int)(blockDim.x >> 5); ++i)
        o |= (static_cast<uint64_t>(s_orw[1][i]) << 32) | s_orw[0][i];
      s_hb = o ? 63 - __clzll(static_cast<long long>(o)) : 0;
      s_prefix = 0;
      s_need = nmiss;
      s_nsel = 0;
    }
    __syncthreads();
    for (int d = (s_hb / 8) * 8; d >= 0; d -= 8) {
      for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      const uint64_t prefix = s_prefix;
      for (int base = 0; base < c.S; base += blockDim.x) {
        const int s = base + tid;
        int digit = -1;
        if (s < c.S) {
          const uint64_t k = skey[s];
          if (k != ~0ull && (d + 8 >= 64 || (k >> (d + 8)) == (prefix >> (d + 8))))
            digit = static_cast<int>((k >> d) & 255u);
        }
        const unsigned same = __match_any_sync(0xffffffffu, digit);
        if (digit >= 0 && lane == __ffs(same) - 1) atomicAdd(&hist[digit], __popc(same));
      }
      __syncthreads();
      if (w == 0) {
        int h[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          h[j] = hist[lane * 8 + j];
          sum += h[j];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int x = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += x;
        }
        const int need = s_need;
        const int excl = incl - sum;
        if (excl < need && need <= incl) {  // the one lane whose bins hold rank `need`
          int run = excl, j = 0;
          while (j < 7 && run + h[j] < need) run += h[j++];
          s_prefix = prefix | (static_cast<uint64_t>(lane * 8 + j) << d);
          s_need = need - run;
        }
      }
      __syncthreads();
    }
    const uint64_t tau = s_prefix;  // the nmiss-th smallest key
    for (int s = tid; s < c.S; s += blockDim.x)
      if (skey[s] <= tau) vsel[atomicAdd(&s_nsel, 1)] = skey[s];
    __syncthreads();
    if (tid < nmiss) {
      const uint64_t k = vsel[tid];
      int r = 0;
      for (int j = 0; j < nmiss; ++j) r += vsel[j] < k;
      vic[r] = k;
    }
    __syncthreads();
  }
  const int64_t clock_new = c.ctr[0] + 1;

  // LRFU: every slot decays by one query before the hits and fills
  if (lrfu && c.lrfu_k)
    for (int s = tid; s < c.S; s += blockDim.x) c.crf[s] -= c.crf[s] >> c.lrfu_k;
  __syncthreads();

  // 4. fills, evictions, recency (and LRFU scores and pins)
  if (tid < nvalid) {
    const int k = qkey[tid];
    const int r = qrank[tid];
    if (r >= 0) {
      const int v = static_cast<int>(vic[r] & ((1u << slot_bits) - 1u));
      const int old = c.slot_key[v];
      if (old >= 0 && old < LE) {
        c.map[old] = -1;
        atomicAdd(&s_evict, 1);
      }
      c.map[k] = v;
      c.slot_key[v] = k;
      c.slot_ts[v] = clock_new;
      miss[3 * r + 0] = k;
      miss[3 * r + 1] = v;
      miss[3 * r + 2] = old;
      if (lrfu) c.crf[v] = kCrfOne;
      if (use_tag) c.pin[v] = use_tag;
    } else {
      const int h = qslot[tid];
      c.slot_ts[h] = clock_new;
      if (lrfu) c.crf[h] = min(c.crf[h] + kCrfOne, kCrfSat);
      if (use_tag) c.pin[h] = use_tag;
    }
    if (record_stats) c.decode_freq[k] += 1;
  }
  __syncthreads();
  if (tid == 0) {
    c.ctr[0] = clock_new;
    if (record_stats) {
      c.ctr[1] += nhit;
      c.ctr[2] += nmiss;
      c.ctr[3] += s_evict;
    }
    *n_miss = nmiss;
  }
}

}  // namespace oes
