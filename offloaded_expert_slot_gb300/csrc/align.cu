// moe_align_block_size for any expert count: a stable counting sort of
// routes by expert in three launches, or in one for up to 1024 routes
// (FreeToken PR #676, Solution and Tests:
// sgl_kernel's single-block count breaks once the experts and the padding
// id no longer fit 1024 threads; each route must be placed exactly once,
// in a block of its own expert; vLLM fork PR #48, What:
// ignore_invalid_experts).
//
//   count:   CTA g histograms its contiguous range of routes -> cnt[g][e]
//            (eight 16-byte loads, 32 routes, in flight a thread)
//   scan:    CTA c takes experts [32c, 32c + 32): its [G x 32] tile of counts
//            in shared memory, scanned over g by all its warps at once;
//            cnt[g][e] becomes the routes of expert e in CTAs before g, and
//            tot[e] the expert's routes
//   scatter: every CTA first scans the padded expert sizes itself (E <= 4096)
//            -> expert offsets; CTA g re-reads its range; each warp counts its
//            segment (16-byte loads), then walks its 32-route groups in order, eight groups' ids loaded at once, and
//            places them by their rank among the group's lanes of the same
//            expert (found with one ballot per bit of the expert id, the
//            eight groups' ballots interleaved), so routes of one expert keep
//            ascending route order (bit-exact, stable); extra CTAs write each
//            expert's block ids and padding, and the unused tail.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "align_dev.cuh"
#include "internal.h"

namespace oes {
namespace {

constexpr int kAlignThreads = 256;  // 8 warps
constexpr int kAlignWarps = kAlignThreads / 32;

struct AlignWs {
  int32_t* cnt;   // [G][E]
  int32_t* off;   // [E] first position of each expert
  int32_t* tot;   // [E] routes of each expert
  int32_t* nblk;  // [1] used blocks
};

constexpr int kAlignUnroll = 8;  // routes (or 32-route groups) loaded at once per thread

__device__ __forceinline__ void count_id(int v, int E, int32_t* hist, bool& bad) {
  if (v >= 0 && v < E) atomicAdd(&hist[v], 1);
  else bad = true;
}

// vec: ids 16-byte aligned; C is a multiple of 256, so every CTA's range
// starts on a 16-byte boundary and is read four ids a load (32 ids in flight
// a thread), its ragged end id by id.
__global__ void __launch_bounds__(kAlignThreads)
    align_count_kernel(const int32_t* __restrict__ ids, int R, int E, int C, int ignore_invalid,
                       int vec, AlignWs ws, int32_t* __restrict__ status) {
  pdl_begin();
  extern __shared__ int32_t hist[];
  const int g = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int r0 = g * C, r1 = min(R, r0 + C);
  const int step = blockDim.x * kAlignUnroll;
  bool bad = false;
  int rs = r0;  // first id the id-by-id loop below counts
  if (vec) {
    const int4* v4 = reinterpret_cast<const int4*>(ids);
    const int q0 = r0 / 4, q1 = r1 / 4;
    for (int qb = q0 + threadIdx.x; qb < q1; qb += step) {
      int4 v[kAlignUnroll];
#pragma unroll
      for (int i = 0; i < kAlignUnroll; ++i) {
        const int q = qb + i * blockDim.x;
        if (q < q1) v[i] = __ldg(v4 + q);
      }
#pragma unroll
      for (int i = 0; i < kAlignUnroll; ++i) {
        if (qb + i * (int)blockDim.x >= q1) continue;  // past the range
        count_id(v[i].x, E, hist, bad);
        count_id(v[i].y, E, hist, bad);
        count_id(v[i].z, E, hist, bad);
        count_id(v[i].w, E, hist, bad);
      }
    }
    rs = q1 * 4;
  }
  for (int rb = rs + threadIdx.x; rb < r1; rb += step) {
    int v[kAlignUnroll];
#pragma unroll
    for (int i = 0; i < kAlignUnroll; ++i) {
      const int r = rb + i * blockDim.x;
      v[i] = (r < r1) ? __ldg(ids + r) : 0;
    }
#pragma unroll
    for (int i = 0; i < kAlignUnroll; ++i) {
      if (rb + i * (int)blockDim.x >= r1) continue;  // past the range
      count_id(v[i], E, hist, bad);
    }
  }
  if (bad && !ignore_invalid) set_status(status, OES_DEV_BAD_ID);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) ws.cnt[(size_t)g * E + e] = hist[e];
}

// CTA c: experts [32c, 32c + 32).  Bands of up to kScanRows rows of the
// [G x 32] tile of per-CTA counts are loaded into shared memory at once (row
// stride 33: no bank conflicts); in a band, warp w sums its rows for the 32
// experts (lane = expert), the warps' sums are scanned, and each warp writes
// its rows' exclusive prefixes back, carrying the band's total to the next.
constexpr int kScanWarps = 32;
constexpr int kScanRows = 1024;
__global__ void __launch_bounds__(32 * kScanWarps)
    align_colscan_kernel(int G, int E, AlignWs ws) {
  pdl_begin();
  extern __shared__ int32_t tile[];  // [min(G, kScanRows)][33]
  __shared__ int32_t band[kScanWarps][33];
  const int c0 = blockIdx.x * 32;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  int carry = 0;  // this lane's expert: routes in the bands before
  for (int gb = 0; gb < G; gb += kScanRows) {
    const int rows = min(kScanRows, G - gb);
    // eight loads in flight a thread (the rows are independent)
    for (int i0 = tid; i0 < rows * 32; i0 += blockDim.x * kAlignUnroll) {
      int x[kAlignUnroll];
#pragma unroll
      for (int u = 0; u < kAlignUnroll; ++u) {
        const int i = i0 + u * (int)blockDim.x, g = i >> 5, j = i & 31;
        x[u] = (i < rows * 32 && c0 + j < E) ? ws.cnt[(size_t)(gb + g) * E + c0 + j] : 0;
      }
#pragma unroll
      for (int u = 0; u < kAlignUnroll; ++u) {
        const int i = i0 + u * (int)blockDim.x;
        if (i < rows * 32) tile[(i >> 5) * 33 + (i & 31)] = x[u];
      }
    }
    __syncthreads();
    const int per = (rows + kScanWarps - 1) / kScanWarps;
    const int g0 = min(rows, w * per), g1 = min(rows, g0 + per);
    int sum = 0;
    for (int g = g0; g < g1; ++g) sum += tile[g * 33 + lane];
    band[w][lane] = sum;
    __syncthreads();
    int run = carry;
    for (int q = 0; q < w; ++q) run += band[q][lane];
    for (int g = g0; g < g1; ++g) {
      const int x = tile[g * 33 + lane];
      if (c0 + lane < E) ws.cnt[(size_t)(gb + g) * E + c0 + lane] = run;
      run += x;
    }
    for (int q = 0; q < kScanWarps; ++q) carry += band[q][lane];
    __syncthreads();  // the tile and band are reused by the next band
  }
  if (w == 0 && c0 + lane < E) ws.tot[c0 + lane] = carry;
}

// Exclusive scan of the padded expert sizes into off[] (shared memory, E <=
// OES_MAX_EXPERTS) by one CTA; returns the padded total.  All threads call it.
__device__ int padded_offsets(const int32_t* __restrict__ tot, int E, int B, int32_t* off,
                              int* warp_tot) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, w = tid >> 5;
  const int per = (E + nt - 1) / nt;
  const int b0 = min(E, tid * per), b1 = min(E, b0 + per);
  int sum = 0;
  for (int e = b0; e < b1; ++e) sum += (tot[e] + B - 1) / B * B;
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
    off[e] = run;
    run += (tot[e] + B - 1) / B * B;
  }
  const int total = warp_tot[(nt >> 5) - 1];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kAlignThreads)
    align_scatter_kernel(const int32_t* __restrict__ ids, int R, int E, int B, int C, int G,
                         int64_t cap, int vec, AlignWs ws, int32_t* __restrict__ sorted_ids,
                         int32_t* __restrict__ block_expert, int32_t* __restrict__ n_post_pad,
                         int32_t* __restrict__ zero, int nzero) {
  pdl_begin();
  extern __shared__ int32_t sm[];
  __shared__ int warp_tot[32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int32_t* off = sm;  // [E] first position of each expert
  const int total = padded_offsets(ws.tot, E, B, off, warp_tot);
  if (blockIdx.x == 0 && threadIdx.x == 0) *n_post_pad = total;
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
  if ((int)blockIdx.x < G) {
    int32_t* wpos = sm + E;  // [kAlignWarps][E]
    const int g = blockIdx.x;
    int nbits = 1;  // bits of the keys: experts 0..E-1, invalid lanes E..E+31
    while ((1 << nbits) < E + 32) ++nbits;
    for (int i = threadIdx.x; i < kAlignWarps * E; i += blockDim.x) wpos[i] = 0;
    __syncthreads();
    const int seg = C / kAlignWarps;
    const int r0 = g * C + w * seg, r1 = min(R, r0 + seg);
    // the warp's counts (order does not matter here): four ids a load when
    // the ids are 16-byte aligned (seg is a multiple of 32 routes, so r0 is
    // a multiple of four), its ragged end id by id
    int rs = r0;
    if (vec) {
      const int4* v4 = reinterpret_cast<const int4*>(ids);
      const int q1 = r1 / 4;
      for (int qb = r0 / 4 + lane; qb < q1; qb += 32 * kAlignUnroll) {
        int4 v[kAlignUnroll];
#pragma unroll
        for (int i = 0; i < kAlignUnroll; ++i) {
          const int q = qb + 32 * i;
          v[i] = (q < q1) ? __ldg(v4 + q) : make_int4(-1, -1, -1, -1);
        }
#pragma unroll
        for (int i = 0; i < kAlignUnroll; ++i) {
          const int x[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (x[j] >= 0 && x[j] < E) atomicAdd(&wpos[w * E + x[j]], 1);
        }
      }
      rs = max(r0, q1 * 4);
    }
    for (int rb = rs + lane; rb < r1; rb += 32 * kAlignUnroll) {
      int v[kAlignUnroll];
#pragma unroll
      for (int i = 0; i < kAlignUnroll; ++i) {
        const int r = rb + 32 * i;
        v[i] = (r < r1) ? __ldg(ids + r) : -1;
      }
#pragma unroll
      for (int i = 0; i < kAlignUnroll; ++i)
        if (v[i] >= 0 && v[i] < E) atomicAdd(&wpos[w * E + v[i]], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int run = off[e] + ws.cnt[(size_t)g * E + e];
      for (int q = 0; q < kAlignWarps; ++q) {
        const int c = wpos[q * E + e];
        wpos[q * E + e] = run;
        run += c;
      }
    }
    __syncthreads();
    for (int rb = r0; rb < r1; rb += 32 * kAlignUnroll) {
      int v[kAlignUnroll];
#pragma unroll
      for (int i = 0; i < kAlignUnroll; ++i) {
        const int r = rb + 32 * i + lane;
        v[i] = (r < r1) ? __ldg(ids + r) : -1;
      }
      // the same-key lanes of all eight groups, bit by bit: eight independent
      // ballots a bit rather than one group's chain of nbits at a time
      int key[kAlignUnroll];
      unsigned grp[kAlignUnroll];
#pragma unroll
      for (int i = 0; i < kAlignUnroll; ++i) {
        key[i] = (v[i] >= 0 && v[i] < E) ? v[i] : E + lane;  // invalid lanes never group
        grp[i] = 0xffffffffu;
      }
      for (int b = 0; b < nbits; ++b) {
#pragma unroll
        for (int i = 0; i < kAlignUnroll; ++i) {
          const bool bit = (key[i] >> b) & 1;
          const unsigned bal = __ballot_sync(0xffffffffu, bit);
          grp[i] &= bit ? bal : ~bal;
        }
      }
#pragma unroll
      for (int i = 0; i < kAlignUnroll; ++i) {
        const int r = rb + 32 * i + lane;
        const bool ok = v[i] >= 0 && v[i] < E;
        const int rank = __popc(grp[i] & ((1u << lane) - 1u));
        if (ok) sorted_ids[wpos[w * E + v[i]] + rank] = r;
        __syncwarp();
        if (ok && rank == 0) wpos[w * E + v[i]] += __popc(grp[i]);
        __syncwarp();
      }
    }
  } else {
    // padding and block experts, expert by expert: expert e owns the blocks
    // [off[e] / B, (off[e] + padded) / B) and pads [off[e] + tot[e],
    // off[e] + padded) with R; past the last block, blocks get -1 and
    // entries R up to the capacity
    const int nblk = total / B;
    const int64_t nb_cap = cap / B;
    const int fill_warps = (gridDim.x - G) * kAlignWarps;
    const int fw = (blockIdx.x - G) * kAlignWarps + w;
    for (int e = fw; e < E; e += fill_warps) {
      const int64_t s0 = off[e], cnt = ws.tot[e];
      const int64_t end = s0 + (cnt + B - 1) / B * B;
      for (int64_t b = s0 / B + lane; b < end / B; b += 32) block_expert[b] = e;
      for (int64_t p = s0 + cnt + lane; p < end; p += 32) sorted_ids[p] = R;
    }
    const int64_t ft = (int64_t)fw * 32 + lane, nft = (int64_t)fill_warps * 32;
    for (int64_t b = nblk + ft; b < nb_cap; b += nft) block_expert[b] = -1;
    for (int64_t p = (int64_t)total + ft; p < cap; p += nft) sorted_ids[p] = R;
  }
}

__global__ void __launch_bounds__(1024)
    align_small_kernel(const int32_t* __restrict__ ids, int R, int E, int B, int64_t cap,
                       int ignore_invalid, int32_t* __restrict__ sorted_ids,
                       int32_t* __restrict__ block_expert, int32_t* __restrict__ n_post_pad,
                       int32_t* __restrict__ status, int32_t* __restrict__ zero, int nzero) {
  pdl_begin();
  extern __shared__ int32_t sm[];
  align_small_cta(ids, R, E, B, cap, ignore_invalid, sorted_ids, block_expert, n_post_pad, status,
                  zero, nzero, sm);
}

// CTA range: a multiple of 256 routes, at least 2048, and about 8 CTAs per
// SM (5 past 1024 experts, where each CTA's zeroing and scan of its warps'
// counters, 8 E of them, weighs more): enough warps to cover the scatter's
// load latency.  Measured at 2^24 routes: 201 -> 163 us over 512 experts
// (2 CTAs per SM before), 223 -> 191 us over 2100.
void align_geometry(int R, int E, int* G, int* C, size_t* ws_bytes) {
  const int sms = num_sms();
  const int per_sm = E <= 1024 ? 8 : 5;
  int64_t c = std::max<int64_t>(2048, ceil_div64(R, (int64_t)sms * per_sm));
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
  const size_t scat_smem = (size_t)(kAlignWarps + 1) * E * 4;
  const size_t scan_smem = (size_t)std::min(G, kScanRows) * 33 * 4;
  if (scat_smem > 48 * 1024) {
    const int rc = set_max_dynamic_smem(reinterpret_cast<const void*>(align_scatter_kernel),
                                        scat_smem, "align_scatter_kernel: shared memory limit");
    if (rc) return rc;
  }
  if (scan_smem > 48 * 1024) {
    const int rc = set_max_dynamic_smem(reinterpret_cast<const void*>(align_colscan_kernel),
                                        scan_smem, "align_colscan_kernel: shared memory limit");
    if (rc) return rc;
  }
  const int vec = ((uintptr_t)ids & 15) == 0 && C % 4 == 0;
  launch_kernel(align_count_kernel, G, kAlignThreads, hist_smem, stream, ids, R, E, C, ignore_invalid,
                vec, ws, status);
  OES_CHECK_LAUNCH("align_count_kernel");
  launch_kernel(align_colscan_kernel, ceil_div(E, 32), 32 * kScanWarps, scan_smem, stream, G, E, ws);
  OES_CHECK_LAUNCH("align_colscan_kernel");
  // fill CTAs: a warp for every four experts (the padding past the last
  // block is at most E * (B - 1) entries)
  const int fill_ctas = (int)std::min<int64_t>(std::max(1, ceil_div(E, kAlignWarps * 4)), (int64_t)num_sms());
  launch_kernel(align_scatter_kernel, G + fill_ctas, kAlignThreads, scat_smem, stream,
      ids, R, E, B, C, G, cap, vec, ws, sorted_ids, block_expert, n_post_pad, zero, nzero);
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
