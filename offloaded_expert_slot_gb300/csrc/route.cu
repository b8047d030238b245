// Routing: gate logits (tiny workload), warp-per-token top-k with softmax
// renormalisation, and the chunk's distinct experts as a fixed-length
// sorted list (FreeToken PR #676, Solution).
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "route_dev.cuh"

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

constexpr int kTopkThreads = 128;

// One warp per token (topk_row).
template <int EPL, typename LT>
__global__ void topk_kernel(const LT* __restrict__ logits, int T, int E, int k,
                            int32_t* __restrict__ ids, float* __restrict__ weights) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps)
    topk_row<EPL, LT>(logits + (size_t)t * E, E, k, lane, ids + (size_t)t * k, weights + (size_t)t * k);
}

// One warp per token (topk_row_filtered), 16-byte loads: E a multiple of V,
// rows 16-byte aligned, E <= 32 * V * Q.  Up to 16 logits a lane the kernel
// fits 48 registers a thread without spilling, so that ten CTAs (40 warps)
// share an SM.
template <int V, int Q, typename LT>
__global__ void __launch_bounds__(kTopkThreads, V * Q <= 16 ? 10 : 1)
    topk_filtered_kernel(const LT* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
                         float* __restrict__ weights) {
  pdl_begin();
  __shared__ uint2 cand[kTopkThreads / 32][33];
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  uint2* my_cand = cand[threadIdx.x >> 5];
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps)
    topk_row_filtered<V, Q, LT>(logits + (size_t)t * E, E, k, lane, ids + (size_t)t * k,
                                weights + (size_t)t * k, my_cand);
}

// Single CTA (distinct_cta).
__global__ void __launch_bounds__(1024)
    distinct_kernel(const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ distinct,
                    int32_t* __restrict__ d_count) {
  pdl_begin();
  extern __shared__ uint8_t flag[];
  distinct_cta(ids, R, E, distinct, d_count, flag);
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
// One wave: as many CTAs as fit on the SMs at once (the kernel loops over
// tokens), at most one warp a token.
template <auto Kernel>
int topk_grid(int T) {
  static const int per_sm = [] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, Kernel, kTopkThreads, 0) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      n = 1;
    }
    return n;
  }();
  return (int)std::min<int64_t>(ceil_div64((int64_t)T * 32, kTopkThreads), (int64_t)num_sms() * per_sm);
}

template <typename LT>
void launch_topk(const LT* logits, int T, int E, int k, int32_t* ids, float* weights,
                 cudaStream_t stream) {
  const int threads = kTopkThreads;
  // the threshold filter with 16-byte loads where the rows allow them
  constexpr int V = 16 / (int)sizeof(LT);
  if (E <= 32 * 32 && E % V == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0) {
    const int q = ceil_div(E, 32 * V);
#define OES_TOPKF(Q)                                                                                   \
  launch_kernel(topk_filtered_kernel<V, Q, LT>, topk_grid<topk_filtered_kernel<V, Q, LT>>(T), threads, 0, \
                stream, logits, T, E, k, ids, weights)
    if (q <= 1) OES_TOPKF(1);
    else if (q <= 2) OES_TOPKF(2);
    else if (q <= 4) OES_TOPKF(4);
    else OES_TOPKF(32 / V);
#undef OES_TOPKF
    return;
  }
  const int epl = ceil_div(E, 32);
#define OES_TOPK(N)                                                                             \
  launch_kernel(topk_kernel<N, LT>, topk_grid<topk_kernel<N, LT>>(T), threads, 0, stream, logits, T, E, \
                k, ids, weights)
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
