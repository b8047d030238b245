// Routing: gate logits (tiny workload), warp-per-token top-k with softmax
// renormalisation, and the chunk's distinct experts as a fixed-length
// sorted list (FreeToken PR #676, Solution).
#include <math.h>

#include <algorithm>

#include "common.cuh"

namespace oes {
namespace {

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// logits[t, e] = sum_h x[t, h] * gate[h, e]; one thread per (t, e), h in order.
__global__ void gate_logits_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ gate,
                                   int T, int H, int E, float* __restrict__ logits) {
  pdl_begin();
  const int t = blockIdx.y;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
    float acc = 0.f;
    const uint16_t* xr = x + (size_t)t * H;
    for (int h = 0; h < H; ++h)
      acc = fmaf(bf16_to_f32(xr[h]), bf16_to_f32(gate[(size_t)h * E + e]), acc);
    logits[(size_t)t * E + e] = acc;
  }
}

__device__ __forceinline__ float load_logit(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_logit(const uint16_t* p) { return bf16_to_f32(__ldg(p)); }

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

// The two best entries (key, position j) of a lane's EPL keys, skipping the
// positions set in `taken`; ties go to the lower j (strict comparisons in
// ascending j).  Position EPL and key 0 mean none.
template <int EPL>
__device__ __forceinline__ void lane_top2(const uint32_t (&key)[EPL], uint32_t taken, uint32_t& k1,
                                          int& j1, uint32_t& k2, int& j2) {
  k1 = k2 = 0u;
  j1 = j2 = EPL;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const uint32_t kj = (j < 32 && ((taken >> (j & 31)) & 1u)) ? 0u : key[j];
    if (kj > k1) {
      k2 = k1;
      j2 = j1;
      k1 = kj;
      j1 = j;
    } else if (kj > k2) {
      k2 = kj;
      j2 = j;
    }
  }
}

// One warp per token.  Lane l holds the keys of experts l, l + 32, ...
// (logits widened to fp32, bf16 exactly) and its two best.  Each of the k
// rounds takes the warp's largest key (one redux.sync), then the lowest
// expert id holding it (another): larger logit first, ties to the lower id.
// Only the winning lane moves on to its next entry: its second best, or, once
// that is used, a rescan of its keys without the taken ones (a bit mask of
// taken positions up to 32 keys a lane; past that the key is cleared).  Lane r keeps
// round r's winner; the weights are a softmax over the k selected logits.
template <int EPL, typename LT>
__global__ void topk_kernel(const LT* __restrict__ logits, int T, int E, int k,
                            int32_t* __restrict__ ids, float* __restrict__ weights) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    const LT* row = logits + (size_t)t * E;
    uint32_t key[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = lane + 32 * j;
      key[j] = (e < E) ? logit_key(load_logit(row + e)) : 0u;
    }
    uint32_t k1, k2;
    int j1, j2;
    lane_top2<EPL>(key, 0u, k1, j1, k2, j2);
    uint32_t taken = 0u;
    bool have2 = true;
    uint32_t my_k = 0u, my_e = 0u;
    for (int r = 0; r < k; ++r) {
      const uint32_t g = __reduce_max_sync(0xffffffffu, k1);
      const uint32_t cand = (k1 == g) ? (uint32_t)(lane + 32 * j1) : 0xffffffffu;
      const uint32_t we = __reduce_min_sync(0xffffffffu, cand);
      if (lane == r) {
        my_k = g;
        my_e = we;
      }
      if (lane == (int)(we & 31u)) {
        if (EPL <= 32) {
          taken |= 1u << (j1 & 31);
        } else {
          // wider rows (more than 1024 experts) clear the taken key in place
#pragma unroll
          for (int j = 0; j < EPL; ++j)
            if (j == j1) key[j] = 0u;
        }
        if (have2) {
          k1 = k2;
          j1 = j2;
          have2 = false;
        } else {
          lane_top2<EPL>(key, taken, k1, j1, k2, j2);
          have2 = true;
        }
      }
    }
    const float my_v = key_logit(my_k);
    const float top = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = (lane < k) ? expf(my_v - top) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < k) {
      ids[(size_t)t * k + lane] = (int32_t)my_e;
      weights[(size_t)t * k + lane] = ex / sum;
    }
  }
}

// Single CTA: presence flags over the E experts, then a block-wide exclusive
// scan turns flags into output positions.
__global__ void __launch_bounds__(1024)
    distinct_kernel(const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ distinct,
                    int32_t* __restrict__ d_count) {
  pdl_begin();
  extern __shared__ uint8_t flag[];
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int i = tid; i < E; i += nt) flag[i] = 0;
  __syncthreads();
  for (int r = tid; r < R; r += nt) {
    const int v = __ldg(ids + r);
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

}  // namespace
}  // namespace oes

using namespace oes;

extern "C" int moe_gate_logits(const uint16_t* x, const uint16_t* gate, int T, int H, int E,
                               float* logits, oes_stream_t stream) {
  OES_REQUIRE(x && gate && logits, "moe_gate_logits: null pointer");
  OES_REQUIRE(T >= 1 && T <= 65535 && H >= 1 && E >= 1 && E <= OES_MAX_EXPERTS,
              "moe_gate_logits: bad sizes T=%d H=%d E=%d", T, H, E);
  const int threads = E < 256 ? ((E + 31) / 32) * 32 : 256;
  dim3 grid(ceil_div(E, threads), T);
  launch_kernel(gate_logits_kernel, grid, threads, 0, stream, x, gate, T, H, E, logits);
  OES_CHECK_LAUNCH("gate_logits_kernel");
  return OES_OK;
}

namespace {
template <typename LT>
void launch_topk(const LT* logits, int T, int E, int k, int32_t* ids, float* weights,
                 cudaStream_t stream) {
  const int threads = 128;
  const int blocks = (int)std::min<int64_t>(ceil_div64((int64_t)T * 32, threads), (int64_t)num_sms() * 16);
  const int epl = ceil_div(E, 32);
#define OES_TOPK(N) \
  launch_kernel(topk_kernel<N, LT>, blocks, threads, 0, stream, logits, T, E, k, ids, weights)
  if (epl <= 1) OES_TOPK(1);
  else if (epl <= 2) OES_TOPK(2);
  else if (epl <= 4) OES_TOPK(4);
  else if (epl <= 8) OES_TOPK(8);
  else if (epl <= 16) OES_TOPK(16);
  else if (epl <= 32) OES_TOPK(32);
  else if (epl <= 64) OES_TOPK(64);
  else OES_TOPK(128);
#undef OES_TOPK
}
}  // namespace

extern "C" int moe_route_topk(const void* logits, int dtype, int T, int E, int k, int32_t* ids,
                              float* weights, oes_stream_t stream) {
  OES_REQUIRE(logits && ids && weights, "moe_route_topk: null pointer");
  OES_REQUIRE(dtype == OES_LOGITS_F32 || dtype == OES_LOGITS_BF16,
              "moe_route_topk: unknown logits type %d", dtype);
  OES_REQUIRE(T >= 0 && E >= 1 && E <= OES_MAX_EXPERTS, "moe_route_topk: bad T=%d E=%d", T, E);
  OES_REQUIRE(k >= 1 && k <= E && k <= OES_MAX_TOPK, "moe_route_topk: bad k=%d (E=%d)", k, E);
  if (T == 0) return OES_OK;
  if (dtype == OES_LOGITS_F32)
    launch_topk(static_cast<const float*>(logits), T, E, k, ids, weights, stream);
  else
    launch_topk(static_cast<const uint16_t*>(logits), T, E, k, ids, weights, stream);
  OES_CHECK_LAUNCH("topk_kernel");
  return OES_OK;
}

extern "C" int moe_distinct_experts(const int32_t* ids, int R, int E, int32_t* distinct,
                                    int32_t* d_count, oes_stream_t stream) {
  OES_REQUIRE(d_count && (R == 0 || (ids && distinct)), "moe_distinct_experts: null pointer");
  OES_REQUIRE(R >= 0 && E >= 1 && E <= OES_MAX_EXPERTS, "moe_distinct_experts: bad R=%d E=%d", R, E);
  launch_kernel(distinct_kernel, 1, 1024, E, stream, ids, R, E, distinct, d_count);
  OES_CHECK_LAUNCH("distinct_kernel");
  return OES_OK;
}
