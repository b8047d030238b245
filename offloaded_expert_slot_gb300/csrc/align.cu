// moe_align_block_size for any expert count: a stable counting sort of
// routes by expert in three launches, or in one for up to 1024 routes
// (FreeToken PR #676, Solution and Tests:
// sgl_kernel's single-block count breaks once the experts and the padding
// id no longer fit 1024 threads; each route must be placed exactly once,
// in a block of its own expert; vLLM fork PR #48, What:
// ignore_invalid_experts).
//
//   count:   CTA g histograms its contiguous range of routes -> cnt[g][e]
//   scan:    one CTA: per expert, its total over CTAs; padded sizes;
//            exclusive scan over experts -> expert offsets; cnt[g][e] becomes
//            the first output position of CTA g's routes of expert e (the
//            expert's offset plus its routes in CTAs before g)
//   scatter: CTA g re-reads its range; each warp walks its 32-route groups
//            in order and places them with __match_any_sync ranks, so routes
//            of one expert keep ascending route order (bit-exact, stable);
//            extra CTAs write the padding and block_expert.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace oes {
namespace {

constexpr int kAlignThreads = 256;  // 8 warps
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kScanBatch = 8;   // per-CTA counts one scan thread loads at once

struct AlignWs {
  int32_t* cnt;   // [G][E]
  int32_t* off;   // [E] first position of each expert
  int32_t* tot;   // [E] routes of each expert
  int32_t* nblk;  // [1] used blocks
};

__global__ void __launch_bounds__(kAlignThreads)
    align_count_kernel(const int32_t* __restrict__ ids, int R, int E, int C, int ignore_invalid,
                       AlignWs ws, int32_t* __restrict__ status) {
  pdl_begin();
  extern __shared__ int32_t hist[];
  const int g = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int r0 = g * C, r1 = min(R, r0 + C);
  bool bad = false;
  for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    const int v = __ldg(ids + r);
    if (v >= 0 && v < E) atomicAdd(&hist[v], 1);
    else bad = true;
  }
  if (bad && !ignore_invalid) set_status(status, OES_DEV_BAD_ID);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) ws.cnt[(size_t)g * E + e] = hist[e];
}

__global__ void __launch_bounds__(1024)
    align_scan_kernel(int G, int E, int B, AlignWs ws, int32_t* __restrict__ n_post_pad,
                      int32_t* __restrict__ zero, int nzero) {
  pdl_begin();
  extern __shared__ int32_t padded[];  // [E]
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, w = tid >> 5;
  for (int i = tid; i < nzero; i += nt) zero[i] = 0;
  // column totals: the loads of a batch are issued together (one round
  // trip per kScanBatch CTAs instead of one per CTA)
  for (int e = tid; e < E; e += nt) {
    int run = 0;
    for (int g0 = 0; g0 < G; g0 += kScanBatch) {
      int c[kScanBatch];
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j) c[j] = (g0 + j < G) ? ws.cnt[(size_t)(g0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j) run += c[j];
    }
    ws.tot[e] = run;
    padded[e] = (run + B - 1) / B * B;
  }
  __syncthreads();
  const int per = (E + nt - 1) / nt;
  const int b0 = min(E, tid * per), b1 = min(E, b0 + per);
  int sum = 0;
  for (int e = b0; e < b1; ++e) sum += padded[e];
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
    int s = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += x;
    }
    if (lane < nw) warp_tot[lane] = s;
  }
  __syncthreads();
  int run = incl - sum + (w ? warp_tot[w - 1] : 0);
  for (int e = b0; e < b1; ++e) {
    ws.off[e] = run;
    run += padded[e];
  }
  const int total = warp_tot[(nt >> 5) - 1];
  if (tid == 0) {
    *n_post_pad = total;
    *ws.nblk = total / B;
  }
  __syncthreads();
  // cnt[g][e] <- offset of expert e + routes of e in CTAs before g
  for (int e = tid; e < E; e += nt) {
    int run = ws.off[e];
    for (int g0 = 0; g0 < G; g0 += kScanBatch) {
      int c[kScanBatch];
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j) c[j] = (g0 + j < G) ? ws.cnt[(size_t)(g0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j) {
        if (g0 + j < G) ws.cnt[(size_t)(g0 + j) * E + e] = run;
        run += c[j];
      }
    }
  }
}

__global__ void __launch_bounds__(kAlignThreads)
    align_scatter_kernel(const int32_t* __restrict__ ids, int R, int E, int B, int C, int G,
                         int64_t cap, AlignWs ws, int32_t* __restrict__ sorted_ids,
                         int32_t* __restrict__ block_expert) {
  pdl_begin();
  extern __shared__ int32_t sm[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if ((int)blockIdx.x < G) {
    int32_t* wpos = sm;  // [kAlignWarps][E]
    const int g = blockIdx.x;
    for (int i = threadIdx.x; i < kAlignWarps * E; i += blockDim.x) wpos[i] = 0;
    __syncthreads();
    const int seg = C / kAlignWarps;
    const int r0 = g * C + w * seg, r1 = min(R, r0 + seg);
    for (int r = r0 + lane; r < r1; r += 32) {
      const int v = __ldg(ids + r);
      if (v >= 0 && v < E) atomicAdd(&wpos[w * E + v], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int run = ws.cnt[(size_t)g * E + e];
      for (int q = 0; q < kAlignWarps; ++q) {
        const int c = wpos[q * E + e];
        wpos[q * E + e] = run;
        run += c;
      }
    }
    __syncthreads();
    for (int rb = r0; rb < r1; rb += 32) {
      const int r = rb + lane;
      const int v = (r < r1) ? __ldg(ids + r) : -1;
      const bool ok = v >= 0 && v < E;
      const int m = ok ? v : -2 - lane;  // invalid lanes never group
      const unsigned grp = __match_any_sync(0xffffffffu, m);
      const int rank = __popc(grp & ((1u << lane) - 1u));
      if (ok) sorted_ids[wpos[w * E + v] + rank] = r;
      __syncwarp();
      if (ok && rank == 0) wpos[w * E + v] += __popc(grp);
      __syncwarp();
    }
  } else {
    // padding and block experts; one warp per block of B entries
    int32_t* off = sm;  // [E]
    for (int e = threadIdx.x; e < E; e += blockDim.x) off[e] = ws.off[e];
    __syncthreads();
    const int nblk = *ws.nblk;
    const int64_t nb_cap = cap / B;
    const int fill_ctas = gridDim.x - G;
    const int fw = (blockIdx.x - G) * kAlignWarps + w;
    for (int64_t b = fw; b < nb_cap; b += (int64_t)fill_ctas * kAlignWarps) {
      int e = -1;
      int64_t first_pad = b * B;
      if (b < nblk) {
        // largest e with off[e] <= b*B
        int lo = 0, hi = E - 1;
        const int x = (int)(b * B);
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (off[mid] <= x) lo = mid;
          else hi = mid - 1;
        }
        e = lo;
        first_pad = (int64_t)off[e] + ws.tot[e];
      }
      if (lane == 0) block_expert[b] = e;
      for (int i = lane; i < B; i += 32) {
        const int64_t p = b * B + i;
        if (p >= first_pad) sorted_ids[p] = R;
      }
    }
  }
}

// The whole align for up to kSmallR routes in one CTA of 1024 threads (a
// decode step's routes: one launch instead of three).  Same output, bit for
// bit: histogram, the padded exclusive scan over experts, each route placed
// at its expert's offset plus the number of earlier routes of that expert
// (counted directly: at most kSmallR^2 / 1024 comparisons a thread), and the
// padding and block experts of every block up to the capacity.
constexpr int kSmallR = 1024;

__global__ void __launch_bounds__(1024)
    align_small_kernel(const int32_t* __restrict__ ids, int R, int E, int B, int64_t cap,
                       int ignore_invalid, int32_t* __restrict__ sorted_ids,
                       int32_t* __restrict__ block_expert, int32_t* __restrict__ n_post_pad,
                       int32_t* __restrict__ status, int32_t* __restrict__ zero, int nzero) {
  pdl_begin();
  for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;           // [E]
  int32_t* off = sm + E;       // [E]
  int32_t* sid = sm + 2 * E;   // [R] expert of each route, -1 if invalid
  __shared__ int warp_tot[32];
  __shared__ int s_total;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, w = tid >> 5;
  for (int e = tid; e < E; e += nt) cnt[e] = 0;
  bool bad = false;
  for (int r = tid; r < R; r += nt) {
    const int v = __ldg(ids + r);
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

// CTA range: a multiple of 256 routes, at least 2048, about 2 CTAs per SM.
void align_geometry(int R, int E, int* G, int* C, size_t* ws_bytes) {
  const int sms = num_sms();
  int64_t c = std::max<int64_t>(2048, ceil_div64(R, (int64_t)sms * 2));
  c = (c + 255) / 256 * 256;
  *C = (int)c;
  *G = std::max(1, (int)ceil_div64(R, c));
  const size_t cnt = (size_t)(*G) * E * 4;
  *ws_bytes = ((cnt + 255) / 256 * 256) + (size_t)E * 8 + 256;
}

}  // namespace
}  // namespace oes

using namespace oes;

extern "C" size_t moe_align_workspace_size(int R, int E, int B) {
  if (R < 0 || E < 1 || B < 1) return 0;
  int G, C;
  size_t ws;
  align_geometry(R, E, &G, &C, &ws);
  return ws;
}

extern "C" int moe_align_block_size(const int32_t* ids, int R, int E, int B, int ignore_invalid,
                                    int32_t* sorted_ids, int32_t* block_expert, int32_t* n_post_pad,
                                    int32_t* status, void* workspace, size_t workspace_bytes,
                                    oes_stream_t stream) {
  return align_run(ids, R, E, B, ignore_invalid, sorted_ids, block_expert, n_post_pad, status,
                   workspace, workspace_bytes, nullptr, 0, stream);
}

namespace oes {
int align_run(const int32_t* ids, int R, int E, int B, int ignore_invalid, int32_t* sorted_ids,
              int32_t* block_expert, int32_t* n_post_pad, int32_t* status, void* workspace,
              size_t workspace_bytes, int32_t* zero, int nzero, cudaStream_t stream) {
  OES_REQUIRE(n_post_pad && workspace && (R == 0 || (ids && sorted_ids && block_expert)),
              "moe_align_block_size: null pointer");
  OES_REQUIRE(nzero >= 0 && (nzero == 0 || zero), "moe_align_block_size: bad words to zero");
  OES_REQUIRE(R >= 0 && R < (1 << 30) && E >= 1 && E <= OES_MAX_EXPERTS && B >= 1 && B <= 1024,
              "moe_align_block_size: bad R=%d E=%d B=%d", R, E, B);
  OES_REQUIRE(((uintptr_t)workspace & 15) == 0, "moe_align_block_size: workspace not 16-byte aligned");
  int G, C;
  size_t need;
  align_geometry(R, E, &G, &C, &need);
  OES_REQUIRE(workspace_bytes >= need, "moe_align_block_size: workspace %zu < %zu bytes",
              workspace_bytes, need);
  const int64_t cap = OES_ALIGN_CAPACITY(R, E, B);
  if (R <= kSmallR) {
    const size_t smem = ((size_t)2 * E + std::max(R, 1)) * 4;  // at most 36 KB
    launch_kernel(align_small_kernel, 1, 1024, smem, stream, ids, R, E, B, cap, ignore_invalid, sorted_ids,
                  block_expert, n_post_pad, status, zero, nzero);
    OES_CHECK_LAUNCH("align_small_kernel");
    return OES_OK;
  }
  uint8_t* p = static_cast<uint8_t*>(workspace);
  AlignWs ws;
  ws.cnt = reinterpret_cast<int32_t*>(p);
  p += ((size_t)G * E * 4 + 255) / 256 * 256;
  ws.off = reinterpret_cast<int32_t*>(p);
  ws.tot = ws.off + E;
  ws.nblk = ws.tot + E;

  const size_t hist_smem = (size_t)E * 4;
  const size_t scat_smem = (size_t)kAlignWarps * E * 4;
  if (scat_smem > 48 * 1024) {
    const int rc = set_max_dynamic_smem(reinterpret_cast<const void*>(align_scatter_kernel),
                                        scat_smem, "align_scatter_kernel: shared memory limit");
    if (rc) return rc;
  }
  launch_kernel(align_count_kernel, G, kAlignThreads, hist_smem, stream, ids, R, E, C, ignore_invalid, ws, status);
  OES_CHECK_LAUNCH("align_count_kernel");
  launch_kernel(align_scan_kernel, 1, 1024, hist_smem, stream, G, E, B, ws, n_post_pad, zero, nzero);
  OES_CHECK_LAUNCH("align_scan_kernel");
  const int fill_ctas = (int)std::min<int64_t>(
      std::max<int64_t>(1, ceil_div64(cap / B, kAlignWarps * 4)), (int64_t)num_sms());
  launch_kernel(align_scatter_kernel, G + fill_ctas, kAlignThreads, scat_smem, stream, 
      ids, R, E, B, C, G, cap, ws, sorted_ids, block_expert);
  OES_CHECK_LAUNCH("align_scatter_kernel");
  return OES_OK;
}
}  // namespace oes

// ------------------------------------------------------ no-allocation variant
// Scratch for moe_align_block_size_noalloc: one fixed buffer per GPU that
// loads the library, held until the process exits.  Host code must not pass
// the symbol itself to a kernel (on the host it names a stand-in, not device
// memory); its device address is looked up once per device below.
static __device__ __align__(256) uint8_t g_align_scratch[OES_ALIGN_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_align_scratch_mu;
void* g_align_scratch_ptr[64] = {nullptr};

// Device address of g_align_scratch on the current device (looked up with
// that device current, on the first call for the device).
int align_scratch_address(void** out) {
  int dev = 0;
  OES_TRY_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) {
    oes::set_error("moe_align_block_size_noalloc: device ordinal %d out of range", dev);
    return OES_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_align_scratch_mu);
  if (!g_align_scratch_ptr[dev]) {
    void* p = nullptr;
    OES_TRY_CUDA(cudaGetSymbolAddress(&p, g_align_scratch));
    g_align_scratch_ptr[dev] = p;
  }
  *out = g_align_scratch_ptr[dev];
  return OES_OK;
}
}  // namespace

extern "C" int moe_align_block_size_noalloc(const int32_t* ids, int R, int E, int B,
                                            int ignore_invalid, int32_t* sorted_ids,
                                            int32_t* block_expert, int32_t* n_post_pad,
                                            int32_t* status, oes_stream_t stream) {
  OES_REQUIRE(R >= 0 && R < (1 << 30) && E >= 1 && E <= OES_MAX_EXPERTS && B >= 1 && B <= 1024,
              "moe_align_block_size_noalloc: bad R=%d E=%d B=%d", R, E, B);
  const size_t need = moe_align_workspace_size(R, E, B);
  if (need > (size_t)OES_ALIGN_NOALLOC_SCRATCH_BYTES) {
    oes::set_error(
        "moe_align_block_size_noalloc: R=%d routes over E=%d experts need %zu bytes of scratch, "
        "more than its fixed %d-byte buffer; call moe_align_block_size with a workspace instead",
        R, E, need, (int)OES_ALIGN_NOALLOC_SCRATCH_BYTES);
    return OES_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  const int rc = align_scratch_address(&scratch);
  if (rc) return rc;
  return moe_align_block_size(ids, R, E, B, ignore_invalid, sorted_ids, block_expert, n_post_pad,
                              status, scratch, (size_t)OES_ALIGN_NOALLOC_SCRATCH_BYTES, stream);
}
