// The grouped SwiGLU expert GEMM over the slot pool, on tcgen05 / TMEM / TMA.
//
// FreeToken PR #676, Solution: a demand chunk reuses the decode GEMM, each
// expert read at its slot, and must give the streamed layer's bytes exactly;
// the expert view knows the layer's expert count, and the NVFP4 prefill
// takes its tiles from routes per expert of the layer, not of the pool.
// vLLM fork PR #48, What: logical alignment plus a physical-row remap.
//
// Design (swap-AB): the weight rows of an expert are the MMA's M side (128
// rows per tile) and the routes of one align block are its N side (the
// block's routes, rounded up to 16), both operands K-major.  One persistent
// kernel template runs both GEMMs:
//   GEMM1 (MODE 1): per (block, 128 intermediate rows): gate and up tiles
//     into two TMEM accumulators, epilogue h = silu(g) * u -> 16-bit h;
//     the block's token rows are gathered from x with 16-byte cp.async
//     copies into the 128-byte-swizzled layout the MMA reads; each lane's
//     copies arrive on the stage's mbarrier when they complete, and the MMA
//     thread orders them before its tensor-core reads with a proxy fence.
//   GEMM2 (MODE 2): per (block, 128 output rows): y = h @ w2^T -> bf16 y
//     at each route's row.
// Warp roles: 0 weight producer (TMA), 1 MMA issuer (one thread), 2 TMEM
// allocator, 3 h producer (GEMM2, TMA), 4-7 epilogue, 8-11 token gather
// (GEMM1, cp.async), and for NVFP4 eight converter warps placed on
// schedulers 0, 2 and 3 (warp id mod 4), so that the scheduler of the MMA
// issuer carries no ALU-heavy warp.
// (NVFP4 only: e2m1 x e4m3 decoded exactly into f16 tiles in shared memory;
// the per-expert fp32 global scale is applied to the fp32 sums).
// The weights of a slot are addressed through a 3-D tensor map over the
// pool [S][rows][K]; the slot coordinate comes from the remap, so the same
// kernel over a contiguous layer buffer (remap = identity) runs the same
// instructions on the same data in the same order: bit-identical output.
// K split (GEMM1, weight-major): when the GEMM1 tiles of the largest routing
// a chunk can have fill at most half the SMs (one token at top-10: 60 tiles
// of 32 K chunks), every tile becomes two units, one per half of its K
// range, on neighbouring CTAs.  Each half leaves its fp32 gate and up sums in
// the workspace; the epilogue warp of the second half to count itself in
// adds half 0 and half 1 and writes h.  The split is part of the plan, so
// every launch of a call, and both paths, take it alike.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "gemm_types.h"
#include "internal.h"

namespace oes {
namespace {

constexpr int kTileM = 128;  // weight rows per MMA
constexpr int kChunkK = 64;  // K elements per pipeline stage (128 bytes of 16-bit)
constexpr int kConvWarps = 8;    // NVFP4 converter warps
constexpr int kConvGroupWarps = kConvWarps / 2;  // two groups take alternate stages
constexpr int kGatherWarps = 4;  // GEMM1 token-gather warps
constexpr int kGatherW0 = 8;     // first gather warp
constexpr int kMaxUnitsPerCta = 256;  // units whose info is tabled in shared memory

// Converter index (0..7) of a warp, or -1: warps 12, 14, 15, 16, 18, 19, 20,
// 22; warps 13, 17 and 21 (the MMA issuer's scheduler) stay idle.
__device__ __forceinline__ int conv_index(int warp) {
  switch (warp) {
    case 12: return 0;
    case 14: return 1;
    case 15: return 2;
    case 16: return 3;
    case 18: return 4;
    case 19: return 5;
    case 20: return 6;
    case 22: return 7;
    default: return -1;
  }
}

__host__ __device__ constexpr int gemm_threads(int wf) { return 32 * (wf ? 23 : 12); }
// token-major kernel: NVFP4 adds 16 converter warps (12..27) in two groups of
// eight that take alternate pipeline stages
constexpr int kTmConvW0 = 12;
constexpr int kTmConvWarps = 16;
constexpr int kTmConvGroupWarps = kTmConvWarps / 2;  // a stage's converter arrivals
__host__ __device__ constexpr int gemm_threads_tm(int wf) { return 32 * (wf ? kTmConvW0 + kTmConvWarps : 12); }

struct Unit {
  int b, m, h, slot, nvalid;  // h: the unit's K half (0 unless the tile's K is split)
  bool skip;
};

constexpr int kFiltered = -2;  // Unit::slot of a block another launch computes

// A routing-table entry: through L2 alone (ld.global.cg) for a kernel that
// reads the tables before its dependency wait (GEMM2, see the kernel), else
// a plain load.
template <bool CG>
__device__ __forceinline__ int32_t ld_tab(const int32_t* p) { return CG ? __ldcg(p) : *p; }
template <bool CG>
__device__ __forceinline__ int32_t ld_tab(const uint8_t* p) { return CG ? __ldcg(p) : *p; }

// Number of routes of block b (padding, value R, only at its end).
template <bool CG>
__device__ __forceinline__ int block_nvalid(const GemmParams& p, int b) {
  const int32_t* s = p.sorted_ids + (int64_t)b * p.BN;
  if (ld_tab<CG>(s + p.BN - 1) < p.R) return p.BN;
  int lo = 0, hi = p.BN - 1;  // first index holding padding
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (ld_tab<CG>(s + mid) < p.R) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Which block / tile a unit is, the slot of its expert, and how many of the
// block's entries are real routes (padding, value R, only at the end).
template <bool CG>
__device__ __forceinline__ Unit unit_info(const GemmParams& p, int u, int nb) {
  // tile index fastest (after the K half): the units of one block run on
  // neighbouring CTAs at the same time, so the block's token rows (GEMM1) or
  // h rows (GEMM2) are read from DRAM once and then served from L2 for its
  // other tiles
  Unit t;
  const int upb = p.n_mtiles * p.ks;  // units per block
  t.b = u / upb;
  t.m = (u % upb) / p.ks;
  t.h = (u % upb) % p.ks;
  const int e = ld_tab<CG>(p.block_expert + t.b);
  const bool valid_e = e >= 0 && e < p.E;
  const bool filtered = p.filter && valid_e && ld_tab<CG>(p.flags + e) != p.filter;
  t.slot = filtered ? kFiltered : (valid_e ? ld_tab<CG>(p.e2s + e) : -1);
  t.nvalid = block_nvalid<CG>(p, t.b);
  t.skip = t.slot < 0 || t.slot >= p.S || t.nvalid == 0;
  return t;
}

__device__ __forceinline__ int round16(int n) { return (n + 15) & ~15; }

// K chunks [kc_lo, kc_hi) of a unit: all of the tile's, or those of its half
__device__ __forceinline__ int kc_lo(const GemmParams& p, const Unit& t) { return t.h * p.n_kc / p.ks; }
__device__ __forceinline__ int kc_hi(const GemmParams& p, const Unit& t) {
  return (t.h + 1) * p.n_kc / p.ks;
}

struct UnitRec {  // shared-memory copy of a Unit; m holds tile * ks + K half
  int b, m, slot, nvalid;
};


// A filtered launch deals out only the units of the selected blocks, densely,
// so that its CTAs get equal shares: the selected block of rank g (blocks in
// order) owns units g * upb + m, upb = n_mtiles * ks (tile fastest after the
// K half, as everywhere), and this
// CTA takes every gridDim.x-th of them into its table.  Every CTA computes the
// same ranks.  Returns the number of units, or -1 when this CTA's share would
// not fit the table (the caller then numbers units as an unfiltered launch and
// skips the filtered ones).  All threads of the CTA call it.
template <bool CG>
__device__ int fill_filtered_units(const GemmParams& p, int nb, UnitRec* utab, int* s_scan) {
  const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int nw = nthr >> 5;
  auto selected = [&](int b) {
    const int e = ld_tab<CG>(p.block_expert + b);
    return e >= 0 && e < p.E && ld_tab<CG>(p.flags + e) == p.filter &&
           ld_tab<CG>(p.sorted_ids + (int64_t)b * p.BN) < p.R;
  };
  if (nb <= nthr) {
    // one block per thread: its expert and its ids, then the expert's group
    // and slot, two rounds of independent loads
    bool sel = false;
    int nvalid = 0, slot = -1;
    if (tid < nb) {
      const int e = ld_tab<CG>(p.block_expert + tid);
      nvalid = block_nvalid<CG>(p, tid);
      if (e >= 0 && e < p.E) {
        const int f = ld_tab<CG>(p.flags + e);
        slot = ld_tab<CG>(p.e2s + e);
        sel = f == p.filter && nvalid > 0;
      }
    }
    const unsigned bal = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) s_scan[warp] = __popc(bal);
    __syncthreads();
    int off = 0, n = 0;
    for (int i = 0; i < nw; ++i) {
      if (i < warp) off += s_scan[i];
      n += s_scan[i];
    }
    const int upb = p.n_mtiles * p.ks;
    const int units = n * upb;
    if (units > kMaxUnitsPerCta * (int)gridDim.x) return -1;
    if (sel) {
      const int g = off + __popc(bal & ((1u << lane) - 1u));
      for (int m = 0; m < upb; ++m) {
        const int v = g * upb + m;
        if (v % (int)gridDim.x == (int)blockIdx.x) utab[v / gridDim.x] = UnitRec{tid, m, slot, nvalid};
      }
    }
    return units;
  }
  int mine = 0;
  for (int b = tid; b < nb; b += nthr) mine += selected(b) ? 1 : 0;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) s_scan[warp] = mine;
  __syncthreads();
  if (tid == 0) {
    int n = 0;
    for (int i = 0; i < nw; ++i) n += s_scan[i];
    s_scan[32] = n;
  }
  __syncthreads();
  const int upb = p.n_mtiles * p.ks;
  const int units = s_scan[32] * upb;
  __syncthreads();
  if (units > kMaxUnitsPerCta * (int)gridDim.x) return -1;
  int base = 0;
  for (int b0 = 0; b0 < nb; b0 += nthr) {
    const int b = b0 + tid;
    const bool sel = b < nb && selected(b);
    const unsigned bal = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) s_scan[warp] = __popc(bal);
    __syncthreads();
    int off = base, chunk = 0;
    for (int i = 0; i < nw; ++i) {
      if (i < warp) off += s_scan[i];
      chunk += s_scan[i];
    }
    if (sel) {
      const int g = off + __popc(bal & ((1u << lane) - 1u));
      const int nvalid = block_nvalid<CG>(p, b);
      const int slot = ld_tab<CG>(p.e2s + ld_tab<CG>(p.block_expert + b));
      for (int m = 0; m < upb; ++m) {
        const int v = g * upb + m;
        if (v % (int)gridDim.x == (int)blockIdx.x) utab[v / gridDim.x] = UnitRec{b, m, slot, nvalid};
      }
    }
    base += chunk;
    __syncthreads();
  }
  return units;
}

// The CTA's u-th unit (u counted in this CTA's sequence), from the table
// filled at kernel start, or computed directly past the table's end.
template <bool CG>
__device__ __forceinline__ Unit my_unit(const GemmParams& p, const UnitRec* tab, int idx, int u, int nb) {
  if (idx < kMaxUnitsPerCta) {
    const UnitRec r = tab[idx];
    Unit t;
    t.b = r.b;
    t.m = r.m / p.ks;
    t.h = r.m % p.ks;
    t.slot = r.slot;
    t.nvalid = r.nvalid;
    t.skip = t.slot < 0 || t.slot >= p.S || t.nvalid == 0;
    return t;
  }
  return unit_info<CG>(p, u, nb);
}

__device__ __forceinline__ uint32_t cvt_e2m1x2_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(r) : "r"(byte));
  return r;
}
// Four e2m1 pairs (one 32-bit word, element 2i in the low nibble of byte i)
// -> four f16x2, byte i -> o[i]; the word is split into bytes by one vector
// move instead of a shift and a narrowing convert per byte.
__device__ __forceinline__ void cvt_e2m1x8_f16x2(uint32_t wd, uint32_t (&o)[4]) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n"
      "  mov.b32 {b0, b1, b2, b3}, %4;\n"
      "  cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      "  cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "  cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      "  cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(wd));
}
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t two) {
  uint32_t r;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(r) : "r"(two));
  return r;
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// f32 pair -> e2m1x2 byte, rounded to nearest even and saturating at 6:
// `hi` in the upper nibble, `lo` in the lower one.
__device__ __forceinline__ uint32_t cvt_f32x2_e2m1x2(float hi, float lo) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// f32 -> e4m3 byte, rounded to nearest even and saturating at 448.
__device__ __forceinline__ uint32_t cvt_f32_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;
}

// W4A4 activations (FreeToken PR #676, Solution: quantised under the max a of
// the layer's input scales).  A block of 16 consecutive values along K
// becomes e2m1 codes q with one e4m3 scale sf: s = amax / (6 a) and
// q_i = v_i / (sf a) in fp32, each rounded to nearest even and saturating;
// a block with sf = 0 is all zero.  The GEMM reads q_i * sf, exact in f16,
// and a multiplies its fp32 sums.
__device__ __forceinline__ uint32_t act_scale_f16x2(float amax, float a, float* sf) {
  const uint32_t sc = cvt_f32_e4m3(__fdiv_rn(amax, __fmul_rn(6.0f, a)));
  const uint32_t sf2 = cvt_e4m3x2_f16x2(sc | (sc << 8));
  *sf = __half2float(__ushort_as_half(static_cast<unsigned short>(sf2 & 0xFFFFu)));
  return sf2;
}
__device__ __forceinline__ void quant16_act(const float (&v)[16], float a, uint32_t (&out)[8]) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  float sf;
  const uint32_t sf2 = act_scale_f16x2(amax, a, &sf);
  const float d = __fmul_rn(sf, a);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t b = sf > 0.0f ? cvt_f32x2_e2m1x2(__fdiv_rn(v[2 * j + 1], d), __fdiv_rn(v[2 * j], d)) : 0u;
    out[j] = hmul2_u32(cvt_e2m1x2_f16x2(b), sf2);
  }
}
// The same for a block spread over 16 consecutive lanes, one value each; all
// 32 lanes of the warp call it.  Returns this lane's f16 q * sf.
__device__ __forceinline__ uint16_t quant_lane_act(float v, float a) {
  float amax = fabsf(v);
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  float sf;
  const uint32_t sf2 = act_scale_f16x2(amax, a, &sf);
  const uint32_t b = sf > 0.0f ? cvt_f32x2_e2m1x2(0.0f, __fdiv_rn(v, __fmul_rn(sf, a))) : 0u;
  return static_cast<uint16_t>(hmul2_u32(cvt_e2m1x2_f16x2(b), sf2) & 0xFFFFu);
}

// One weight row of one K chunk: 32 bytes of e2m1 pairs and a 32-bit word of
// four e4m3 scales (one per 16 elements) -> 64 f16 = 8 x 16 bytes, stored at
// the 128-byte-swizzled position of row `row` of a K-major tile.  Every
// product e2m1 * e4m3 has at most 6 significant bits and lies in
// [2^-10, 2688], so it is exact in f16.
__device__ __forceinline__ void convert_row(const uint8_t* q, uint32_t scales, uint8_t* tile,
                                            int row) {
  const uint4 q0 = *reinterpret_cast<const uint4*>(q);
  const uint4 q1 = *reinterpret_cast<const uint4*>(q + 16);
  const uint32_t s01 = cvt_e4m3x2_f16x2(scales & 0xFFFFu);
  const uint32_t s23 = cvt_e4m3x2_f16x2(scales >> 16);
  const uint32_t sc[4] = {__byte_perm(s01, 0, 0x1010), __byte_perm(s01, 0, 0x3232),
                          __byte_perm(s23, 0, 0x1010), __byte_perm(s23, 0, 0x3232)};
  const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  uint8_t* rowp = tile + row * 128;
  const int sw = row & 7;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t wd = words[c];
    const uint32_t s = sc[c >> 1];
    uint32_t f[4];
    cvt_e2m1x8_f16x2(wd, f);
    uint4 o;
    o.x = hmul2_u32(f[0], s);
    o.y = hmul2_u32(f[1], s);
    o.z = hmul2_u32(f[2], s);
    o.w = hmul2_u32(f[3], s);
    *reinterpret_cast<uint4*>(rowp + ((c ^ sw) << 4)) = o;
  }
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// GEMM1 epilogue of weight row i for routes c0 .. c0 + C - 1 of the unit's
// block: h = silu(g gs) * (u gs) from the fp32 sums g and u, stored as 16-bit
// h.  W4A4 quantises h per 16 rows, one row a lane: all 32 lanes take part.
template <int WF, int C>
__device__ __forceinline__ void store_h(const GemmParams& p, const Unit& t, int i, int c0,
                                        const float (&g)[C], const float (&v)[C], float gs) {
  if (WF && p.a4) {
#pragma unroll
    for (int j = 0; j < C; ++j) {
      const int n = c0 + j;
      const bool keep = i < p.I && n < t.nvalid;
      const float hv = keep ? silu(g[j] * gs) * (v[j] * gs) : 0.0f;
      const uint16_t hb = quant_lane_act(hv, p.act[1]);
      if (keep) p.h[((int64_t)t.b * p.BN + n) * p.I + i] = hb;
    }
  } else if (i < p.I) {
#pragma unroll
    for (int j = 0; j < C; ++j) {
      const int n = c0 + j;
      if (n < t.nvalid) {
        const float gv = g[j] * gs;
        const float uv = v[j] * gs;
        const float hv = silu(gv) * uv;
        uint16_t hb;
        if (WF) hb = __half_as_ushort(__float2half_rn(hv));
        else hb = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
        p.h[((int64_t)t.b * p.BN + n) * p.I + i] = hb;
      }
    }
  }
}

template <int MODE, int WF>
__global__ void __launch_bounds__(gemm_threads(WF), 1)
    grouped_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  constexpr int kA = (MODE == 1) ? 2 : 1;  // weight tiles per stage (gate + up, or w2)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int a_bytes = kA * kTileM * 128;
  const int b_bytes = p.BN * 128;
  const int stage_bytes = a_bytes + b_bytes;
  const int rq_bytes = kA * kTileM * 32;
  const int rs_bytes = kA * kTileM * 4;
  const int raw_stage = ((rq_bytes + rs_bytes) + 1023) & ~1023;
  uint8_t* stages = smem;
  uint8_t* raw = stages + p.NS * stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw + (WF ? p.NR * raw_stage : 0));
  uint64_t* full = bars;
  uint64_t* empty = full + p.NS;
  uint64_t* rfull = empty + p.NS;
  uint64_t* rempty = rfull + p.NR;
  uint64_t* tfull = rempty + p.NR;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 2);
  UnitRec* utab = reinterpret_cast<UnitRec*>(tmem_holder + 4);  // [kMaxUnitsPerCta]

  // set-up that reads and writes no global memory runs before the wait for
  // the previous kernel: barrier initialisation and the tensor-map prefetch
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      // arrivals per stage: the weight side (TMA producer, or the converter
      // warps) and the token side (32 gather lanes, or the h TMA producer)
      mbar_init(&full[s], (WF ? kConvGroupWarps : 1) + (MODE == 1 ? 32 * kGatherWarps : 1));
      mbar_init(&empty[s], 1);
    }
    for (int r = 0; r < p.NR; ++r) {
      mbar_init(&rfull[r], 1);
      mbar_init(&rempty[r], kConvGroupWarps);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if (MODE == 2) tma_prefetch_desc(&maps.b);
    if (WF) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.sc);
    } else {
      tma_prefetch_desc(&maps.a);
    }
  }
  // GEMM1 waits here for the kernels before it.  GEMM2 is launched while
  // GEMM1 runs (GEMM1 releases it after its set-up): everything GEMM2 reads
  // but h -- the routing tables, the groups, the slot map and the weights --
  // was complete before GEMM1 passed this wait, so GEMM2 builds its unit
  // table, takes TMEM and streams its first weight stages now, and only the
  // h producer waits for GEMM1 to complete.  Its table reads go to L2
  // (ld.global.cg), not to a possibly stale L1 line.
  if (MODE == 1) pdl_wait();
  // a filtered launch over a group with no experts has nothing to do
  if (p.filter && p.gcount && ld_tab<MODE == 2>(p.gcount + p.filter) == 0) return;

  const int nb = ld_tab<MODE == 2>(p.n_post_pad) / p.BN;
  int total = nb * p.n_mtiles * p.ks;
  const uint32_t acc_cols = (MODE == 1) ? 2 * p.BN : p.BN;
  __shared__ int s_scan[33];
  const int dense = p.filter ? fill_filtered_units<MODE == 2>(p, nb, utab, s_scan) : -1;
  if (dense >= 0) {
    total = dense;
  } else {
    // every thread looks up one of this CTA's units (independent loads in
    // parallel), so the roles below never wait on global memory for them
    for (int i = threadIdx.x; i < kMaxUnitsPerCta; i += blockDim.x) {
      const int u = blockIdx.x + i * gridDim.x;
      if (u >= total) break;
      const Unit t = unit_info<MODE == 2>(p, u, nb);
      utab[i] = UnitRec{t.b, t.m * p.ks + t.h, t.slot, t.nvalid};
    }
  }
  __syncthreads();
  // a CTA without units leaves before it takes TMEM (a small or filtered
  // launch leaves most CTAs idle)
  if ((int)blockIdx.x >= total) return;

  if (warp == 2) {
    tmem_alloc(tmem_holder, p.tmem_cols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // A GEMM1 of at most two units a CTA lets GEMM2, the next kernel on its
  // stream, launch now: GEMM2's CTAs take the SMs this launch leaves idle or
  // frees and set up while it runs (see the wait above).  A longer GEMM1
  // does not: CTAs of GEMM2 resident early would hold the SMs its CTAs free
  // against kernels of other streams that have work before GEMM2 can start.
  if (MODE == 1 && total <= 2 * (int)gridDim.x) pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------- weight producer
      int s = 0, ph = 0, r = 0, rph = 0;
      bool ok = true;
      for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
        const Unit t = my_unit<MODE == 2>(p, utab, ui, u, nb);
        if (t.skip) continue;
        const int row0 = t.m * kTileM;
        for (int kc = kc_lo(p, t), ke = kc_hi(p, t); kc < ke && ok; ++kc) {
          if (!WF) {
            ok = mbar_wait(&empty[s], ph ^ 1, p.status);
            if (!ok) break;
            uint8_t* A = stages + s * stage_bytes;
            mbar_arrive_expect_tx(&full[s], a_bytes);
            tma_load_3d(A, &maps.a, &full[s], kc * kChunkK, row0, t.slot);
            if (MODE == 1)
              tma_load_3d(A + kTileM * 128, &maps.a, &full[s], kc * kChunkK, p.up_row0 + row0,
                          t.slot);
            if (++s == p.NS) { s = 0; ph ^= 1; }
          } else {
            ok = mbar_wait(&rempty[r], rph ^ 1, p.status);
            if (!ok) break;
            uint8_t* Q = raw + r * raw_stage;
            uint8_t* SC = Q + rq_bytes;
            mbar_arrive_expect_tx(&rfull[r], rq_bytes + rs_bytes);
            tma_load_3d(Q, &maps.q, &rfull[r], kc * (kChunkK / 2), row0, t.slot);
            tma_load_3d(SC, &maps.sc, &rfull[r], row0, kc, t.slot);
            if (MODE == 1) {
              tma_load_3d(Q + kTileM * 32, &maps.q, &rfull[r], kc * (kChunkK / 2),
                          p.up_row0 + row0, t.slot);
              tma_load_3d(SC + kTileM * 4, &maps.sc, &rfull[r], p.up_row0 + row0, kc, t.slot);
            }
            if (++r == p.NR) { r = 0; rph ^= 1; }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      int s = 0, ph = 0;
      uint32_t use[2] = {0, 0};
      int a = 0;
      bool ok = true;
      for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
        const Unit t = my_unit<MODE == 2>(p, utab, ui, u, nb);
        if (t.skip) continue;
        const uint32_t N = round16(t.nvalid);
        const uint32_t idesc = idesc_f16(WF ? 0u : 1u, kTileM, N);
        ok = mbar_wait(&tempty[a], (use[a] & 1) ^ 1, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + a * acc_cols;
        const int k0 = kc_lo(p, t), k1 = kc_hi(p, t);
        for (int kc = k0; kc < k1; ++kc) {
          ok = mbar_wait(&full[s], ph, p.status);
          if (!ok) break;
          tc_fence_after();
          if (MODE == 1) fence_proxy_async_smem();  // cp.async-written tokens -> tensor core
          const uint32_t A = smem_u32(stages + s * stage_bytes);
          // +32 bytes along K = +2 in the descriptor's start-address field
          const uint64_t ad = smem_desc_sw128(A);
          const uint64_t ud = smem_desc_sw128(A + kTileM * 128);
          const uint64_t bd = smem_desc_sw128(A + a_bytes);
#pragma unroll
          for (int kk = 0; kk < kChunkK / 16; ++kk) {
            const uint32_t acc = (kc != k0 || kk) ? 1u : 0u;
            tc_mma_f16(d0, ad + 2 * kk, bd + 2 * kk, idesc, acc);
            if (MODE == 1) tc_mma_f16(d0 + p.BN, ud + 2 * kk, bd + 2 * kk, idesc, acc);
          }
          tc_commit(&empty[s]);
          if (++s == p.NS) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        tc_commit(&tfull[a]);
        ++use[a];
        a ^= 1;
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------ h producer (GEMM2)
    if (MODE == 2 && lane == 0) {
      pdl_wait();  // h is GEMM1's output
      int s = 0, ph = 0;
      bool ok = true;
      for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
        const Unit t = my_unit<MODE == 2>(p, utab, ui, u, nb);
        if (t.skip) continue;
        for (int kc = kc_lo(p, t), ke = kc_hi(p, t); kc < ke; ++kc) {
          ok = mbar_wait(&empty[s], ph ^ 1, p.status);
          if (!ok) break;
          uint8_t* B = stages + s * stage_bytes + a_bytes;
          mbar_arrive_expect_tx(&full[s], b_bytes);
          tma_load_2d(B, &maps.b, &full[s], kc * kChunkK, t.b * p.BN);
          if (++s == p.NS) { s = 0; ph ^= 1; }
        }
      }
    }
  } else if (warp >= kGatherW0 && warp < kGatherW0 + kGatherWarps) {
    // ----------------------------------------------- token gather (GEMM1)
    // 128 threads; thread g copies 16-byte chunk (g & 7) of rows
    // (g >> 3) + 16 j of the block's tokens.  Each thread's copies arrive on
    // the stage's full barrier when they complete (no thread waits for them).
    if (MODE == 1) {
      const int g = threadIdx.x - kGatherW0 * 32;
      const int c = g & 7, r0 = g >> 3;
      int s = 0, ph = 0;
      bool ok = true;
      for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
        const Unit t = my_unit<MODE == 2>(p, utab, ui, u, nb);
        if (t.skip) continue;
        const int N = round16(t.nvalid);
        int64_t src_off[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int n = r0 + 16 * j;
          const int tk = (n < t.nvalid) ? p.sorted_ids[(int64_t)t.b * p.BN + n] / p.k : 0;
          src_off[j] = (int64_t)tk * p.H * 2 + c * 16;
        }
        for (int kc = kc_lo(p, t), ke = kc_hi(p, t); kc < ke; ++kc) {
          if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1, p.status);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          const uint32_t b_s = smem_u32(stages + s * stage_bytes + a_bytes);
          const uint8_t* xg = reinterpret_cast<const uint8_t*>(p.xg) + kc * (kChunkK * 2);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int n = r0 + 16 * j;
            if (n < N) cp_async16(b_s + n * 128 + ((c ^ (n & 7)) << 4), xg + src_off[j]);
          }
          cp_async_mbar_arrive(&full[s]);
          if (++s == p.NS) { s = 0; ph ^= 1; }
        }
      }
      cp_async_wait_all();  // no copy of this thread outlives the CTA
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;  // TMEM lane = weight row within the tile
    uint32_t use[2] = {0, 0};
    int a = 0;
    bool ok = true;
    for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
      const Unit t = my_unit<MODE == 2>(p, utab, ui, u, nb);
      if (t.skip) {
        if (MODE == 2 && t.nvalid > 0 && t.slot != kFiltered) {
          // an expert without a slot: its routes get zeros (and a status bit)
          const int col = t.m * kTileM + row;
          if (col < p.H)
            for (int n = 0; n < t.nvalid; ++n)
              p.y[(int64_t)p.sorted_ids[(int64_t)t.b * p.BN + n] * p.H + col] = 0;
          if (row == 0) set_status(p.status, OES_DEV_BAD_ID);
        }
        continue;
      }
      ok = mbar_wait(&tfull[a], use[a] & 1, p.status);
      if (!ok) break;
      tc_fence_after();
      float gs = 1.0f;
      if (WF)
        gs = *reinterpret_cast<const float*>(p.pool + (int64_t)t.slot * p.row_bytes + p.scal_off +
                                             (MODE == 1 ? 0 : 4));
      if (WF && p.a4) gs *= p.act[MODE - 1];
      const uint32_t tl = tmem_base + ((uint32_t)(q * 32) << 16) + a * acc_cols;
      const int N = round16(t.nvalid);
      if (MODE == 1 && p.ks == 2) {
        // K split: each epilogue warp puts its 32 rows of this half's fp32
        // sums in the tile's part and counts itself in; the warp of the
        // second half to get there adds half 0's and half 1's sums and
        // writes those rows of h.  No warp waits for another.
        const int64_t tile = (int64_t)t.b * p.n_mtiles + t.m;
        const int64_t hsz = 2 * (int64_t)p.BN * kTileM;  // gate and up sums of one half
        const float* const tp = p.part + tile * 2 * hsz + row;  // this lane's row, half 0
        float* wg = p.part + (tile * 2 + t.h) * hsz + row;
        float* wu = wg + (int64_t)p.BN * kTileM;
#pragma unroll 1
        for (int c0 = 0; c0 < N; c0 += 16, wg += 16 * kTileM, wu += 16 * kTileM) {
          uint32_t g[16], v[16];
          tmem_ld_16(tl + c0, g);
          tmem_ld_16(tl + p.BN + c0, v);
          tc_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            wg[j * kTileM] = __uint_as_float(g[j]);
            wu[j * kTileM] = __uint_as_float(v[j]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[a]);  // the accumulator is free again
        ++use[a];
        a ^= 1;
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atom_add_acq_rel_gpu(p.tcount + tile * 4 + q, 1) == 1;
        // the warp barrier orders lane 0's acquire before the other lanes'
        // reads of the other half's sums below
        __syncwarp();
        if (!__shfl_sync(0xffffffffu, last, 0)) continue;
        __threadfence();
        const int64_t uo = (int64_t)p.BN * kTileM;
#pragma unroll 1
        for (int c0 = 0; c0 < N; c0 += 8) {  // 8 routes at a time: fewer loads in flight
          const float* r0 = tp + (int64_t)c0 * kTileM;
          const float* r1 = r0 + hsz;
          float gf[8], vf[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            gf[j] = __ldcg(r0 + j * kTileM) + __ldcg(r1 + j * kTileM);
            vf[j] = __ldcg(r0 + uo + j * kTileM) + __ldcg(r1 + uo + j * kTileM);
          }
          store_h<WF, 8>(p, t, t.m * kTileM + row, c0, gf, vf, gs);
        }
        continue;
      }
      for (int c0 = 0; c0 < N; c0 += 16) {
        uint32_t g[16];
        tmem_ld_16(tl + c0, g);
        if (MODE == 1) {
          uint32_t v[16];
          tmem_ld_16(tl + p.BN + c0, v);
          tc_wait_ld();
          float gf[16], vf[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            gf[j] = __uint_as_float(g[j]);
            vf[j] = __uint_as_float(v[j]);
          }
          store_h<WF, 16>(p, t, t.m * kTileM + row, c0, gf, vf, gs);
        } else {
          tc_wait_ld();
          const int col = t.m * kTileM + row;
          if (col < p.H) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = c0 + j;
              if (n < t.nvalid) {
                const int r = p.sorted_ids[(int64_t)t.b * p.BN + n];
                const float yv = __uint_as_float(g[j]) * gs;
                p.y[(int64_t)r * p.H + col] = __bfloat16_as_ushort(__float2bfloat16_rn(yv));
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[a]);
      ++use[a];
      a ^= 1;
    }
  } else if (WF && conv_index(warp) >= 0) {
    // --------------------------------------------------- NVFP4 converters
    // Two groups of four warps take alternate K chunks, so that one group's
    // hand-off of a stage to the MMA (proxy fence, arrivals, the next
    // waits) overlaps the other group's conversion.  NS and NR are even, so
    // every stage and raw stage is always used by the same group, and a
    // group never waits on a barrier phase the other group has yet to
    // release.  Thread rr of a group converts row rr of each 128-row tile:
    // GEMM1's gate and up rows rr, GEMM2's row rr.
    const int ci = conv_index(warp);
    const int group = ci / kConvGroupWarps;
    const int rr = (ci % kConvGroupWarps) * 32 + lane;
    int s = 0, ph = 0, r = 0, rph = 0, n = 0;
    bool ok = true;
    for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
      const Unit t = my_unit<MODE == 2>(p, utab, ui, u, nb);
      if (t.skip) continue;
      for (int kc = kc_lo(p, t), ke = kc_hi(p, t); kc < ke; ++kc, ++n) {
        if ((n & 1) == group) {
          ok = mbar_wait(&rfull[r], rph, p.status) && mbar_wait(&empty[s], ph ^ 1, p.status);
          if (!ok) break;
          const uint8_t* Q = raw + r * raw_stage;
          const uint32_t* SC = reinterpret_cast<const uint32_t*>(Q + rq_bytes);
          uint8_t* A = stages + s * stage_bytes;
#pragma unroll
          for (int a = 0; a < kA; ++a)
            convert_row(Q + (a * kTileM + rr) * 32, SC[a * kTileM + rr], A + a * kTileM * 128, rr);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&rempty[r]);
            mbar_arrive(&full[s]);
          }
        }
        if (++r == p.NR) { r = 0; rph ^= 1; }
        if (++s == p.NS) { s = 0; ph ^= 1; }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}


// ---------------------------------------------------------------------------
// Token-major variant, for blocks of 128 routes (many routes per expert): the
// block's 128 token rows are the MMA's M side and a 256-row weight tile its N
// side (GEMM1: 128 gate rows + the matching 128 up rows; GEMM2: 256 rows of
// w2), so one 128 x 256 x 16 MMA per K step replaces two 128 x N x 16 ones.
// TMEM: two 256-column fp32 accumulators; thread = token row in the
// epilogue, which stores h / y rows with 16-byte vectors.  Same roles,
// barriers and shared-memory stage layout as the kernel above (weights at
// the stage start, 32 KB; tokens after them, 16 KB).
// At most 64 registers a thread: the NVFP4 variant has 28 warps, 7 on each
// of the SM's four sub-partitions, and at 72 registers they would leave 256
// registers of a sub-partition free, too few for the miss-copy warp that
// runs beside this kernel; the copy's CTAs then waited for GEMM CTAs to exit
// and were packed onto the few SMs that freed first (a 2.5x slower copy).
// At 64 nothing spills.
template <int MODE, int WF>
__global__ void __maxnreg__(64)
    grouped_gemm_tm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  constexpr int kN = 256;                  // weight rows per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int w_bytes = kN * 128;            // 32 KB of 16-bit weights per K chunk
  const int x_bytes = kTileM * 128;        // 16 KB of 16-bit tokens per K chunk
  const int stage_bytes = w_bytes + x_bytes;
  const int rq_bytes = kN * 32;
  const int rs_bytes = kN * 4;
  const int raw_stage = ((rq_bytes + rs_bytes) + 1023) & ~1023;
  uint8_t* stages = smem;
  uint8_t* raw = stages + p.NS * stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw + (WF ? p.NR * raw_stage : 0));
  uint64_t* full = bars;
  uint64_t* empty = full + p.NS;
  uint64_t* rfull = empty + p.NS;
  uint64_t* rempty = rfull + p.NR;
  uint64_t* tfull = rempty + p.NR;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 2);
  UnitRec* utab = reinterpret_cast<UnitRec*>(tmem_holder + 4);

  pdl_wait();
  // a filtered launch over a group with no experts has nothing to do
  if (p.filter && p.gcount && p.gcount[p.filter] == 0) return;

  const int nb = *p.n_post_pad / p.BN;
  int total = nb * p.n_mtiles * p.ks;
  __shared__ int s_scan[33];
  const int dense = p.filter ? fill_filtered_units<false>(p, nb, utab, s_scan) : -1;
  if (dense >= 0) {
    total = dense;
  } else {
    for (int i = threadIdx.x; i < kMaxUnitsPerCta; i += blockDim.x) {
      const int u = blockIdx.x + i * gridDim.x;
      if (u >= total) break;
      const Unit t = unit_info<false>(p, u, nb);
      utab[i] = UnitRec{t.b, t.m * p.ks + t.h, t.slot, t.nvalid};
    }
  }
  __syncthreads();
  // a CTA without units leaves before it sets up barriers or takes TMEM
  // (a small or filtered launch leaves most CTAs idle)
  if ((int)blockIdx.x >= total) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(&full[s], (WF ? kTmConvGroupWarps : 1) + (MODE == 1 ? 32 * kGatherWarps : 1));
      mbar_init(&empty[s], 1);
    }
    for (int r = 0; r < p.NR; ++r) {
      mbar_init(&rfull[r], 1);
      mbar_init(&rempty[r], kTmConvGroupWarps);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if (MODE == 2) tma_prefetch_desc(&maps.b);
    if (WF) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.sc);
    } else {
      tma_prefetch_desc(&maps.a);
    }
  }

  if (warp == 2) {
    tmem_alloc(tmem_holder, p.tmem_cols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  // weight rows of tile j: GEMM1 gate [128j, +128) and up [I + 128j, +128);
  // GEMM2 w2 rows [256j, +256)
  auto row_a = [&](int j) { return (MODE == 1) ? j * kTileM : j * kN; };
  auto row_b = [&](int j) { return (MODE == 1) ? p.up_row0 + j * kTileM : j * kN + kTileM; };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------- weight producer
      int s = 0, ph = 0, r = 0, rph = 0;
      bool ok = true;
      for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
        const Unit t = my_unit<false>(p, utab, ui, u, nb);
        if (t.skip) continue;
        const int ra = row_a(t.m), rb = row_b(t.m);
        for (int kc = 0; kc < p.n_kc && ok; ++kc) {
          if (!WF) {
            ok = mbar_wait(&empty[s], ph ^ 1, p.status);
            if (!ok) break;
            uint8_t* W = stages + s * stage_bytes;
            mbar_arrive_expect_tx(&full[s], w_bytes);
            tma_load_3d(W, &maps.a, &full[s], kc * kChunkK, ra, t.slot);
            tma_load_3d(W + kTileM * 128, &maps.a, &full[s], kc * kChunkK, rb, t.slot);
            if (++s == p.NS) { s = 0; ph ^= 1; }
          } else {
            ok = mbar_wait(&rempty[r], rph ^ 1, p.status);
            if (!ok) break;
            uint8_t* Q = raw + r * raw_stage;
            uint8_t* SC = Q + rq_bytes;
            mbar_arrive_expect_tx(&rfull[r], rq_bytes + rs_bytes);
            tma_load_3d(Q, &maps.q, &rfull[r], kc * (kChunkK / 2), ra, t.slot);
            tma_load_3d(Q + kTileM * 32, &maps.q, &rfull[r], kc * (kChunkK / 2), rb, t.slot);
            tma_load_3d(SC, &maps.sc, &rfull[r], ra, kc, t.slot);
            tma_load_3d(SC + kTileM * 4, &maps.sc, &rfull[r], rb, kc, t.slot);
            if (++r == p.NR) { r = 0; rph ^= 1; }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      int s = 0, ph = 0;
      uint32_t use[2] = {0, 0};
      int a = 0;
      bool ok = true;
      const uint32_t idesc = idesc_f16(WF ? 0u : 1u, kTileM, kN);
      for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
        const Unit t = my_unit<false>(p, utab, ui, u, nb);
        if (t.skip) continue;
        ok = mbar_wait(&tempty[a], (use[a] & 1) ^ 1, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + a * kN;
        for (int kc = 0; kc < p.n_kc; ++kc) {
          ok = mbar_wait(&full[s], ph, p.status);
          if (!ok) break;
          tc_fence_after();
          if (MODE == 1) fence_proxy_async_smem();  // cp.async-written tokens -> tensor core
          const uint32_t W = smem_u32(stages + s * stage_bytes);
          const uint64_t wd = smem_desc_sw128(W);             // B: 256 weight rows
          const uint64_t xd = smem_desc_sw128(W + w_bytes);   // A: 128 token rows
#pragma unroll
          for (int kk = 0; kk < kChunkK / 16; ++kk)
            tc_mma_f16(d0, xd + 2 * kk, wd + 2 * kk, idesc, (kc | kk) ? 1u : 0u);
          tc_commit(&empty[s]);
          if (++s == p.NS) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        tc_commit(&tfull[a]);
        ++use[a];
        a ^= 1;
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------ h producer (GEMM2)
    if (MODE == 2 && lane == 0) {
      int s = 0, ph = 0;
      bool ok = true;
      for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
        const Unit t = my_unit<false>(p, utab, ui, u, nb);
        if (t.skip) continue;
        for (int kc = 0; kc < p.n_kc; ++kc) {
          ok = mbar_wait(&empty[s], ph ^ 1, p.status);
          if (!ok) break;
          uint8_t* X = stages + s * stage_bytes + w_bytes;
          mbar_arrive_expect_tx(&full[s], x_bytes);
          tma_load_2d(X, &maps.b, &full[s], kc * kChunkK, t.b * p.BN);
          if (++s == p.NS) { s = 0; ph ^= 1; }
        }
      }
    }
  } else if (warp >= kGatherW0 && warp < kGatherW0 + kGatherWarps) {
    // ----------------------------------------------- token gather (GEMM1)
    if (MODE == 1) {
      const int g = threadIdx.x - kGatherW0 * 32;
      const int c = g & 7, r0 = g >> 3;
      int s = 0, ph = 0;
      bool ok = true;
      for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
        const Unit t = my_unit<false>(p, utab, ui, u, nb);
        if (t.skip) continue;
        const int N = round16(t.nvalid);
        int64_t src_off[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int n = r0 + 16 * j;
          const int tk = (n < t.nvalid) ? p.sorted_ids[(int64_t)t.b * p.BN + n] / p.k : 0;
          src_off[j] = (int64_t)tk * p.H * 2 + c * 16;
        }
        for (int kc = 0; kc < p.n_kc; ++kc) {
          if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1, p.status);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          const uint32_t x_s = smem_u32(stages + s * stage_bytes + w_bytes);
          const uint8_t* xg = reinterpret_cast<const uint8_t*>(p.xg) + kc * (kChunkK * 2);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int n = r0 + 16 * j;
            if (n < N) cp_async16(x_s + n * 128 + ((c ^ (n & 7)) << 4), xg + src_off[j]);
          }
          cp_async_mbar_arrive(&full[s]);
          if (++s == p.NS) { s = 0; ph ^= 1; }
        }
      }
      cp_async_wait_all();
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;  // TMEM lane = token row of the block
    uint32_t use[2] = {0, 0};
    int a = 0;
    bool ok = true;
    for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
      const Unit t = my_unit<false>(p, utab, ui, u, nb);
      const bool live = row < t.nvalid;
      if (t.skip) {
        if (MODE == 2 && live && t.slot != kFiltered) {
          const int r = p.sorted_ids[(int64_t)t.b * p.BN + row];
          for (int c = 0; c < kN; c += 8) {
            const int col = t.m * kN + c;
            if (col < p.H) *reinterpret_cast<uint4*>(p.y + (int64_t)r * p.H + col) = make_uint4(0, 0, 0, 0);
          }
          if (row == 0) set_status(p.status, OES_DEV_BAD_ID);
        }
        continue;
      }
      ok = mbar_wait(&tfull[a], use[a] & 1, p.status);
      if (!ok) break;
      tc_fence_after();
      float gs = 1.0f;
      if (WF)
        gs = *reinterpret_cast<const float*>(p.pool + (int64_t)t.slot * p.row_bytes + p.scal_off +
                                             (MODE == 1 ? 0 : 4));
      if (WF && p.a4) gs *= p.act[MODE - 1];
      const uint32_t tl = tmem_base + ((uint32_t)(q * 32) << 16) + a * kN;
      if (MODE == 1) {
        uint16_t* hrow = p.h + ((int64_t)t.b * p.BN + row) * p.I;
        for (int c0 = 0; c0 < kTileM; c0 += 16) {
          uint32_t g[16], v[16];
          tmem_ld_16(tl + c0, g);
          tmem_ld_16(tl + kTileM + c0, v);
          tc_wait_ld();
          const int i0 = t.m * kTileM + c0;
          if (live && i0 < p.I) {
            uint32_t packed[8];
            if (WF && p.a4) {
              float hv[16];
#pragma unroll
              for (int j = 0; j < 16; ++j)
                hv[j] = silu(__uint_as_float(g[j]) * gs) * (__uint_as_float(v[j]) * gs);
              quant16_act(hv, p.act[1], packed);
            } else {
#pragma unroll
              for (int j = 0; j < 16; j += 2) {
                float h0 = silu(__uint_as_float(g[j]) * gs) * (__uint_as_float(v[j]) * gs);
                float h1 = silu(__uint_as_float(g[j + 1]) * gs) * (__uint_as_float(v[j + 1]) * gs);
                uint32_t lo, hi;
                if (WF) {
                  lo = __half_as_ushort(__float2half_rn(h0));
                  hi = __half_as_ushort(__float2half_rn(h1));
                } else {
                  lo = __bfloat16_as_ushort(__float2bfloat16_rn(h0));
                  hi = __bfloat16_as_ushort(__float2bfloat16_rn(h1));
                }
                packed[j / 2] = lo | (hi << 16);
              }
            }
            uint4* dst = reinterpret_cast<uint4*>(hrow + i0);
            dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
          }
        }
      } else {
        const int r = live ? p.sorted_ids[(int64_t)t.b * p.BN + row] : 0;
        uint16_t* yrow = p.y + (int64_t)r * p.H;
        for (int c0 = 0; c0 < kN; c0 += 16) {
          uint32_t g[16];
          tmem_ld_16(tl + c0, g);
          tc_wait_ld();
          const int col = t.m * kN + c0;
          if (live && col < p.H) {
            uint32_t packed[8];
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(g[j]) * gs));
              const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(g[j + 1]) * gs));
              packed[j / 2] = lo | (hi << 16);
            }
            uint4* dst = reinterpret_cast<uint4*>(yrow + col);
            dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[a]);
      ++use[a];
      a ^= 1;
    }
  } else if (WF && warp >= kTmConvW0) {
    // --------------------------------------------------- NVFP4 converters
    // group 0 converts the even pipeline stages, group 1 the odd ones; in a
    // group, thread rr converts weight row rr of the 256-row tile
    const int group = (warp - kTmConvW0) >> 3;
    const int rr = ((warp - kTmConvW0) & 7) * 32 + lane;
    int s = 0, ph = 0, r = 0, rph = 0, n = 0;
    bool ok = true;
    for (int u = blockIdx.x, ui = 0; u < total && ok; u += gridDim.x, ++ui) {
      const Unit t = my_unit<false>(p, utab, ui, u, nb);
      if (t.skip) continue;
      for (int kc = 0; kc < p.n_kc; ++kc, ++n) {
        if ((n & 1) == group) {
          ok = mbar_wait(&rfull[r], rph, p.status) && mbar_wait(&empty[s], ph ^ 1, p.status);
          if (!ok) break;
          const uint8_t* Q = raw + r * raw_stage;
          const uint32_t* SC = reinterpret_cast<const uint32_t*>(Q + rq_bytes);
          uint8_t* W = stages + s * stage_bytes;
          convert_row(Q + rr * 32, SC[rr], W + (rr / kTileM) * kTileM * 128, rr & (kTileM - 1));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&rempty[r]);
            mbar_arrive(&full[s]);
          }
        }
        if (++r == p.NR) { r = 0; rph ^= 1; }
        if (++s == p.NS) { s = 0; ph ^= 1; }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

// f16 copy of x for the NVFP4 path (its MMAs run on f16 operands).
__global__ void x_to_f16_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ x16,
                                int64_t n) {
  pdl_wait();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float f = __uint_as_float(static_cast<uint32_t>(x[i]) << 16);
    x16[i] = __half_as_ushort(__float2half_rn(f));
  }
}

// W4A4: act[0] = max of the layer's w13 input scales, act[1] = max of its w2
// input scales (one CTA).  A non-positive or non-finite maximum is flagged
// OES_DEV_BAD_ID and replaced by 1.
__global__ void act_scale_kernel(const float* __restrict__ in13, const float* __restrict__ in2,
                                 int E, float* __restrict__ act, int32_t* __restrict__ status) {
  pdl_begin();
  __shared__ float red[2][32];
  float m13 = -INFINITY, m2 = -INFINITY;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    m13 = fmaxf(m13, in13[e]);
    m2 = fmaxf(m2, in2[e]);
  }
  for (int o = 16; o >= 1; o >>= 1) {
    m13 = fmaxf(m13, __shfl_xor_sync(0xffffffffu, m13, o));
    m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    red[0][w] = m13;
    red[1][w] = m2;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) {
      m13 = fmaxf(m13, red[0][i]);
      m2 = fmaxf(m2, red[1][i]);
    }
    const bool ok = m13 > 0.0f && m2 > 0.0f && isfinite(m13) && isfinite(m2);
    if (!ok) set_status(status, OES_DEV_BAD_ID);
    act[0] = ok ? m13 : 1.0f;
    act[1] = ok ? m2 : 1.0f;
  }
}

// W4A4: x [T, H] bf16 -> x16 [T, H] f16 holding q * sf per block of 16 along H.
__global__ void x_quant_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ x16,
                               int64_t nblk, const float* __restrict__ act) {
  pdl_wait();
  const float a = act[0];
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nblk;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(x + i * 16);
    const uint4 b0 = src[0], b1 = src[1];
    const uint32_t w[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    float v[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[2 * j] = __uint_as_float(w[j] << 16);
      v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
    uint32_t o[8];
    quant16_act(v, a, o);
    uint4* dst = reinterpret_cast<uint4*>(x16 + i * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// out[t, :] = sum_{j=0..k-1} w[t, j] * y[t*k + j, :], fp32 in j order -> bf16.
constexpr int kCombineBatch = 8;
__global__ void combine_kernel(const uint16_t* __restrict__ y, const float* __restrict__ w,
                               const int32_t* __restrict__ ids, int T, int k, int H, int E,
                               uint16_t* __restrict__ out) {
  pdl_wait();
  const int vec = H / 8;
  const int64_t n = (int64_t)T * vec;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = static_cast<int>(i / vec);
    const int c = static_cast<int>(i % vec);
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    // eight routes' rows are loaded together (every y row exists, so the
    // loads need not wait for the ids), then added in j order, skipping
    // routes outside [0, E)
    for (int j0 = 0; j0 < k; j0 += kCombineBatch) {
      uint4 v[kCombineBatch];
      float wj[kCombineBatch];
      bool ok[kCombineBatch];
#pragma unroll
      for (int b = 0; b < kCombineBatch; ++b) {
        const int j = j0 + b;
        ok[b] = false;
        if (j < k) {
          const int e = ids[(int64_t)t * k + j];
          ok[b] = e >= 0 && e < E;
          wj[b] = w[(int64_t)t * k + j];
          v[b] = *reinterpret_cast<const uint4*>(y + ((int64_t)t * k + j) * H + c * 8);
        }
      }
#pragma unroll
      for (int b = 0; b < kCombineBatch; ++b) {
        if (!ok[b]) continue;
        const uint32_t u[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[2 * q] = fmaf(wj[b], __uint_as_float(u[q] << 16), acc[2 * q]);
          acc[2 * q + 1] = fmaf(wj[b], __uint_as_float(u[q] & 0xFFFF0000u), acc[2 * q + 1]);
        }
      }
    }
    uint4 o;
    uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * q]));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * q + 1]));
      op[q] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(out + (int64_t)t * H + c * 8) = o;
  }
}

struct Sections {
  int64_t w13, w2, w13q, w13s, w2q, w2s, scal;
};

Sections sections(int wfmt, int H, int I) {
  Sections s{};
  if (wfmt == OES_WFMT_BF16) {
    s.w13 = 0;
    s.w2 = (int64_t)2 * I * H * 2;
  } else {
    s.w13q = 0;
    s.w13s = s.w13q + (int64_t)2 * I * H / 2;
    s.w2q = s.w13s + (int64_t)2 * I * H / 16;
    s.w2s = s.w2q + (int64_t)H * I / 2;
    s.scal = s.w2s + (int64_t)H * I / 16;
  }
  return s;
}

int64_t expected_row_bytes(int wfmt, int H, int I) {
  if (wfmt == OES_WFMT_BF16) return (int64_t)6 * H * I;
  return sections(wfmt, H, I).scal + 16;
}

struct Ws {
  uint16_t* h;
  uint16_t* y;
  uint16_t* x16;
  float* act;        // W4A4: the layer's two activation scales
  float* part;       // GEMM1 K split: fp32 sums of each tile's halves
  int32_t* tcount;   // GEMM1 K split: halves finished per tile and epilogue warp
  size_t bytes;
};

// GEMM1 tiles of the largest routing a chunk of R routes can have (blocks of
// 16, the weight-major kernel), if few enough that splitting their K range
// could pay: then the workspace holds the split's sums.  0 otherwise.
constexpr int64_t kSplitMaxTiles = 128;
int64_t split_tiles(int64_t R, int E, int I, int B) {
  if (B != 16 || R == 0) return 0;
  const int64_t tiles = OES_ALIGN_CAPACITY(R, E, B) / B * ((I + kTileM - 1) / kTileM);
  return tiles <= kSplitMaxTiles ? tiles : 0;
}

Ws carve(void* base, int T, int k, int E, int H, int I, int B, int wfmt) {
  Ws w{};
  const int64_t R = (int64_t)T * k;
  const int64_t cap = OES_ALIGN_CAPACITY(R, E, B);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  size_t off = 0;
  uint8_t* p = static_cast<uint8_t*>(base);
  w.h = reinterpret_cast<uint16_t*>(p + off);
  off += up((size_t)cap * I * 2);
  w.y = reinterpret_cast<uint16_t*>(p + off);
  off += up((size_t)R * H * 2);
  w.x16 = reinterpret_cast<uint16_t*>(p + off);
  if (wfmt != OES_WFMT_BF16) off += up((size_t)T * H * 2);
  w.act = reinterpret_cast<float*>(p + off);
  if (wfmt == OES_WFMT_NVFP4_W4A4) off += 256;
  const int64_t st = split_tiles(R, E, I, B);
  w.part = reinterpret_cast<float*>(p + off);
  off += up((size_t)st * 2 * 2 * B * kTileM * 4);
  w.tcount = reinterpret_cast<int32_t*>(p + off);
  off += up((size_t)st * 4 * 4);
  w.bytes = off + 256;
  return w;
}

int smem_plan(int MODE, int wf, int BN, int* NS, int* NR, size_t* bytes) {
  const int kA = MODE == 1 ? 2 : 1;
  const int stage = kA * kTileM * 128 + BN * 128;
  const int raw_stage = ((kA * kTileM * 36) + 1023) / 1024 * 1024;
  const int budget = 200 * 1024 - kMaxUnitsPerCta * (int)sizeof(UnitRec);
  // NVFP4: even ring sizes, one stage in two for each converter group
  const int nr = wf ? (MODE == 1 ? 4 : 8) : 0;
  int ns = std::min(8, (budget - nr * raw_stage) / stage);
  if (wf) ns &= ~1;
  if (ns < 2) return OES_ERR_UNSUPPORTED;
  *NS = ns;
  *NR = wf ? nr : 1;
  *bytes = 1024 + (size_t)ns * stage + (size_t)nr * raw_stage +
           (size_t)(2 * ns + 2 * (*NR) + 4) * 8 + 16 + (size_t)kMaxUnitsPerCta * sizeof(UnitRec) + 64;
  return OES_OK;
}

int smem_plan_tm(int wf, int* NS, int* NR, size_t* bytes) {
  const int stage = 256 * 128 + kTileM * 128;
  const int raw_stage = 9 * 1024;
  const int budget = 220 * 1024 - kMaxUnitsPerCta * (int)sizeof(UnitRec);
  const int nr = wf ? 8 : 0;
  const int ns = std::min(6, (budget - nr * raw_stage) / stage);
  if (ns < 2) return OES_ERR_UNSUPPORTED;
  *NS = ns;
  *NR = wf ? nr : 1;
  *bytes = 1024 + (size_t)ns * stage + (size_t)nr * raw_stage + (size_t)(2 * ns + 2 * (*NR) + 4) * 8 +
           16 + (size_t)kMaxUnitsPerCta * sizeof(UnitRec) + 64;
  return OES_OK;
}

template <int MODE, int WF>
int launch_gemm_tm(const GemmMaps& maps, const GemmParams& p0, cudaStream_t stream) {
  GemmParams p = p0;
  size_t smem;
  int rc = smem_plan_tm(WF, &p.NS, &p.NR, &smem);
  if (rc) {
    set_error("grouped GEMM (token-major): no pipeline fits");
    return rc;
  }
  p.tmem_cols = 512;
  if ((rc = set_max_dynamic_smem(reinterpret_cast<const void*>(grouped_gemm_tm_kernel<MODE, WF>),
                                  smem, "grouped_gemm_tm_kernel: shared memory limit")))
    return rc;
  launch_kernel(grouped_gemm_tm_kernel<MODE, WF>, num_sms(), gemm_threads_tm(WF), smem, stream, maps, p);
  OES_CHECK_LAUNCH("grouped_gemm_tm_kernel");
  return OES_OK;
}

template <int MODE, int WF>
int launch_gemm(const GemmMaps& maps, const GemmParams& p0, int BN, cudaStream_t stream) {
  GemmParams p = p0;
  size_t smem;
  int rc = smem_plan(MODE, WF, BN, &p.NS, &p.NR, &smem);
  if (rc) {
    set_error("grouped GEMM: no pipeline fits BN=%d", BN);
    return rc;
  }
  p.tmem_cols = (MODE == 1) ? 4 * BN : 2 * BN;
  if (p.tmem_cols < 32) p.tmem_cols = 32;
  if ((rc = set_max_dynamic_smem(reinterpret_cast<const void*>(grouped_gemm_kernel<MODE, WF>), smem,
                                  "grouped_gemm_kernel: shared memory limit")))
    return rc;
  launch_kernel(grouped_gemm_kernel<MODE, WF>, num_sms(), gemm_threads(WF), smem, stream, maps, p);
  OES_CHECK_LAUNCH("grouped_gemm_kernel");
  return OES_OK;
}

}  // namespace

int tile_plan(int R, int E) {
  // routes per expert of the LAYER: up to 8, blocks of 16 routes on the
  // weight-major kernel; more, blocks of 128 routes on the token-major one
  const int per = (R + E - 1) / std::max(E, 1);
  return per <= 8 ? 16 : 128;
}

}  // namespace oes

using namespace oes;

extern "C" int oes_tile_plan(int R, int E, int* block) {
  OES_REQUIRE(block && R >= 0 && E >= 1, "oes_tile_plan: bad arguments");
  *block = tile_plan(R, E);
  return OES_OK;
}

extern "C" size_t moe_grouped_gemm_workspace_size(const oes_routed_experts* v, int T, int k) {
  if (!v || T < 0 || k < 1 || v->E < 1) return 0;
  const int B = tile_plan(T * k, v->E);
  return carve(nullptr, T, k, v->E, v->H, v->I, B, v->wfmt).bytes;
}

extern "C" int moe_grouped_gemm_workspace_views(const oes_routed_experts* v, int T, int k,
                                                void* workspace, uint16_t** h, uint16_t** y,
                                                uint16_t** x16) {
  OES_REQUIRE(v && workspace && T >= 0 && k >= 1 && v->E >= 1,
              "moe_grouped_gemm_workspace_views: bad arguments");
  const Ws ws = carve(workspace, T, k, v->E, v->H, v->I, tile_plan(T * k, v->E), v->wfmt);
  if (h) *h = ws.h;
  if (y) *y = ws.y;
  if (x16) *x16 = v->wfmt == OES_WFMT_BF16 ? nullptr : ws.x16;
  return OES_OK;
}

namespace oes {

// Validates the call and builds the tensor maps and kernel parameters of both
// GEMMs, on the host only: nothing is launched, so a composite call can
// validate its GEMM before it changes any state.  gemm_prepare_x then writes
// the GEMMs' 16-bit copy of x (NVFP4 weights).
int gemm_prepare(const oes_routed_experts* v, const uint16_t* x, int T, int k,
                 const int32_t* sorted_ids, const int32_t* block_expert, const int32_t* n_post_pad,
                 int B, void* workspace, size_t workspace_bytes, int32_t* status, GemmPlan* g) {
  OES_REQUIRE(v && x && sorted_ids && block_expert && n_post_pad && workspace && v->pool && v->e2s,
              "moe_grouped_gemm_slots: null pointer");
  const int E = v->E, H = v->H, I = v->I, S = v->S;
  OES_REQUIRE(E >= 1 && E <= OES_MAX_EXPERTS && S >= 1, "moe_grouped_gemm_slots: bad E=%d S=%d", E, S);
  OES_REQUIRE(H >= 64 && I >= 64 && H % 64 == 0 && I % 64 == 0 && H <= 16384 && I <= 16384,
              "moe_grouped_gemm_slots: H=%d I=%d must be multiples of 64 in [64, 16384]", H, I);
  OES_REQUIRE(v->wfmt == OES_WFMT_BF16 || v->wfmt == OES_WFMT_NVFP4 ||
                  v->wfmt == OES_WFMT_NVFP4_W4A4,
              "moe_grouped_gemm_slots: bad wfmt");
  OES_REQUIRE(v->wfmt != OES_WFMT_NVFP4_W4A4 || (v->input_scale13 && v->input_scale2),
              "moe_grouped_gemm_slots: W4A4 needs the layer's input scales in the view");
  OES_REQUIRE(T >= 0 && T <= (1 << 24) && k >= 1 && k <= OES_MAX_TOPK,
              "moe_grouped_gemm_slots: bad T=%d k=%d", T, k);
  const int64_t need_row = expected_row_bytes(v->wfmt, H, I);
  OES_REQUIRE(v->row_bytes >= need_row && v->row_bytes % 16 == 0,
              "moe_grouped_gemm_slots: row_bytes %lld (layout needs %lld, multiple of 16)",
              (long long)v->row_bytes, (long long)need_row);
  OES_REQUIRE(((uintptr_t)v->pool & 15) == 0 && ((uintptr_t)x & 15) == 0,
              "moe_grouped_gemm_slots: pool and x must be 16-byte aligned");
  const int R = T * k;
  const int plan = tile_plan(R, E);
  OES_REQUIRE(B == plan, "moe_grouped_gemm_slots: block %d differs from the tile plan %d (R=%d, E=%d)",
              B, plan, R, E);
  g->empty = (T == 0);
  if (g->empty) return OES_OK;
  OES_REQUIRE(((uintptr_t)workspace & 255) == 0, "moe_grouped_gemm_slots: workspace not 256-byte aligned");
  const Ws ws = carve(workspace, T, k, E, H, I, B, v->wfmt);
  OES_REQUIRE(workspace_bytes >= ws.bytes, "moe_grouped_gemm_slots: workspace %zu < %zu bytes",
              workspace_bytes, ws.bytes);
  const int64_t cap = OES_ALIGN_CAPACITY(R, E, B);
  const Sections sec = sections(v->wfmt, H, I);
  const uint8_t* pool = static_cast<const uint8_t*>(v->pool);
  const int wf = v->wfmt != OES_WFMT_BF16;
  const int a4 = v->wfmt == OES_WFMT_NVFP4_W4A4;
  g->wf = wf;
  g->tm = (B == 128);  // token-major kernel for blocks of 128 routes
  g->y = ws.y;
  g->T = T;
  g->k = k;
  g->H = H;
  g->E = E;

  GemmMaps m1{}, m2{};
  int rc;
  const uint16_t* xb = x;
  g->a4 = a4;
  g->x = x;
  g->x16 = ws.x16;
  g->act = ws.act;
  g->in13 = v->input_scale13;
  g->in2 = v->input_scale2;
  g->status = status;
  if (wf) xb = ws.x16;
  const CUtensorMapDataType t16 = wf ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  {
    const uint64_t dims[2] = {(uint64_t)I, (uint64_t)cap};
    const uint64_t str[1] = {(uint64_t)I * 2};
    const uint32_t box[2] = {64, (uint32_t)B};
    if ((rc = encode_tiled(&m2.b, t16, 2, ws.h, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))) return rc;
  }
  const uint64_t rb = (uint64_t)v->row_bytes;
  if (!wf) {
    const uint32_t box[3] = {64, 128, 1};
    const uint64_t d1[3] = {(uint64_t)H, (uint64_t)2 * I, (uint64_t)S}, s1[2] = {(uint64_t)H * 2, rb};
    if ((rc = encode_tiled(&m1.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pool + sec.w13, d1, s1, box,
                           CU_TENSOR_MAP_SWIZZLE_128B)))
      return rc;
    const uint64_t d2[3] = {(uint64_t)I, (uint64_t)H, (uint64_t)S}, s2[2] = {(uint64_t)I * 2, rb};
    if ((rc = encode_tiled(&m2.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pool + sec.w2, d2, s2, box,
                           CU_TENSOR_MAP_SWIZZLE_128B)))
      return rc;
  } else {
    const uint32_t qbox[3] = {32, 128, 1}, sbox[3] = {128, 1, 1};
    const uint64_t dq1[3] = {(uint64_t)H / 2, (uint64_t)2 * I, (uint64_t)S}, sq1[2] = {(uint64_t)H / 2, rb};
    if ((rc = encode_tiled(&m1.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, pool + sec.w13q, dq1, sq1, qbox,
                           CU_TENSOR_MAP_SWIZZLE_NONE)))
      return rc;
    const uint64_t ds1[3] = {(uint64_t)2 * I, (uint64_t)H / 64, (uint64_t)S},
                   ss1[2] = {(uint64_t)2 * I * 4, rb};
    if ((rc = encode_tiled(&m1.sc, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, pool + sec.w13s, ds1, ss1, sbox,
                           CU_TENSOR_MAP_SWIZZLE_NONE)))
      return rc;
    const uint64_t dq2[3] = {(uint64_t)I / 2, (uint64_t)H, (uint64_t)S}, sq2[2] = {(uint64_t)I / 2, rb};
    if ((rc = encode_tiled(&m2.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, pool + sec.w2q, dq2, sq2, qbox,
                           CU_TENSOR_MAP_SWIZZLE_NONE)))
      return rc;
    const uint64_t ds2[3] = {(uint64_t)H, (uint64_t)I / 64, (uint64_t)S}, ss2[2] = {(uint64_t)H * 4, rb};
    if ((rc = encode_tiled(&m2.sc, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, pool + sec.w2s, ds2, ss2, sbox,
                           CU_TENSOR_MAP_SWIZZLE_NONE)))
      return rc;
  }

  GemmParams p{};
  p.sorted_ids = sorted_ids;
  p.block_expert = block_expert;
  p.n_post_pad = n_post_pad;
  p.e2s = v->e2s;
  p.flags = nullptr;
  p.filter = 0;
  p.pool = pool;
  p.row_bytes = v->row_bytes;
  p.scal_off = sec.scal;
  p.R = R;
  p.k = k;
  p.BN = B;
  p.H = H;
  p.I = I;
  p.E = E;
  p.S = S;
  p.up_row0 = I;
  p.ks = 1;
  p.xg = xb;
  p.a4 = a4;
  p.act = ws.act;
  p.h = ws.h;
  p.y = ws.y;
  p.status = status;
  g->m1 = m1;
  g->m2 = m2;
  g->p1 = p;
  g->p1.n_mtiles = ceil_div(I, kTileM);
  g->p1.n_kc = H / kChunkK;
  g->p2 = p;
  g->p2.n_mtiles = g->tm ? ceil_div(H, 256) : ceil_div(H, kTileM);
  g->p2.n_kc = I / kChunkK;
  // GEMM1's K split: when the tiles of the largest routing this chunk can
  // have fill at most half the SMs (a one-token decode), each tile's K range
  // is shared by two CTAs.  Decided from the plan alone, so every launch of
  // a call, and the slot and streamed paths, split alike.
  const int64_t st = split_tiles(R, E, I, B);
  g->split_tiles = 0;
  if (!g->tm && st > 0 && st * 2 <= num_sms() && g->p1.n_kc >= 2) {
    g->split_tiles = (int)st;
    g->p1.ks = 2;
    g->p1.part = ws.part;
    g->p1.tcount = ws.tcount;
  }
  g->counters = ws.tcount;
  g->n_counters = g->split_tiles * 4;
  return OES_OK;
}

// The x kernels of a prepared GEMM: the f16 copy of x (NVFP4 weights), or for
// W4A4 the layer's activation scales and the quantised x.
int gemm_prepare_x(const GemmPlan& g, cudaStream_t stream) {
  if (g.empty || !g.wf) return OES_OK;
  const int64_t n = (int64_t)g.T * g.H;
  if (g.a4) {
    launch_kernel(act_scale_kernel, 1, 256, 0, stream, g.in13, g.in2, g.E, g.act, g.status);
    OES_CHECK_LAUNCH("act_scale_kernel");
    const int64_t nblk = n / 16;
    const int blocks = (int)std::min<int64_t>(ceil_div64(nblk, 256), (int64_t)num_sms() * 8);
    launch_kernel(x_quant_kernel, blocks, 256, 0, stream, g.x, g.x16, nblk, g.act);
    OES_CHECK_LAUNCH("x_quant_kernel");
  } else {
    const int blocks = (int)std::min<int64_t>(ceil_div64(n, 256), (int64_t)num_sms() * 8);
    launch_kernel(x_to_f16_kernel, blocks, 256, 0, stream, g.x, g.x16, n);
    OES_CHECK_LAUNCH("x_to_f16_kernel");
  }
  return OES_OK;
}

// GEMM1 then GEMM2 over the blocks `filter` selects (flags: device [E]
// group of each expert; filter 0 = every block).
int gemm_run(const GemmPlan& g, int filter, const uint8_t* flags, const int32_t* gcount,
             cudaStream_t stream) {
  if (g.empty) return OES_OK;
  GemmParams p1 = g.p1, p2 = g.p2;
  p1.filter = p2.filter = filter;
  p1.flags = p2.flags = flags;
  p1.gcount = p2.gcount = gcount;
  const int B = p1.BN;
  int rc;
  if (g.tm) rc = g.wf ? launch_gemm_tm<1, 1>(g.m1, p1, stream) : launch_gemm_tm<1, 0>(g.m1, p1, stream);
  else rc = g.wf ? launch_gemm<1, 1>(g.m1, p1, B, stream) : launch_gemm<1, 0>(g.m1, p1, B, stream);
  if (rc) return rc;
  if (g.tm) rc = g.wf ? launch_gemm_tm<2, 1>(g.m2, p2, stream) : launch_gemm_tm<2, 0>(g.m2, p2, stream);
  else rc = g.wf ? launch_gemm<2, 1>(g.m2, p2, B, stream) : launch_gemm<2, 0>(g.m2, p2, B, stream);
  return rc;
}

int gemm_combine(const GemmPlan& g, const int32_t* ids, const float* weights, uint16_t* out,
                 cudaStream_t stream) {
  if (g.empty) return OES_OK;
  OES_REQUIRE(ids && weights && out && ((uintptr_t)out & 15) == 0,
              "moe_grouped_gemm_slots: ids, weights and a 16-byte aligned out are required");
  const int64_t nvec = (int64_t)g.T * (g.H / 8);
  launch_kernel(combine_kernel, (int)std::min<int64_t>(ceil_div64(nvec, 256), (int64_t)num_sms() * 8), 256, 0, stream, g.y, weights, ids, g.T, g.k, g.H, g.E, out);
  OES_CHECK_LAUNCH("combine_kernel");
  return OES_OK;
}

}  // namespace oes

extern "C" int moe_grouped_gemm_slots(const oes_routed_experts* v, const uint16_t* x, int T, int k,
                                      const int32_t* ids, const float* weights,
                                      const int32_t* sorted_ids, const int32_t* block_expert,
                                      const int32_t* n_post_pad, int B, void* workspace,
                                      size_t workspace_bytes, uint16_t* out, int32_t* status,
                                      oes_stream_t stream) {
  OES_REQUIRE(ids && weights && out, "moe_grouped_gemm_slots: null pointer");
  GemmPlan g;
  int rc = gemm_prepare(v, x, T, k, sorted_ids, block_expert, n_post_pad, B, workspace,
                        workspace_bytes, status, &g);
  if (rc) return rc;
  const GemmCounters sc = gemm_counters(g);
  if (sc.n > 0) OES_TRY_CUDA(cudaMemsetAsync(sc.ptr, 0, (size_t)sc.n * 4, stream));
  if ((rc = gemm_prepare_x(g, stream))) return rc;
  if ((rc = gemm_run(g, 0, nullptr, nullptr, stream))) return rc;
  return gemm_combine(g, ids, weights, out, stream);
}
