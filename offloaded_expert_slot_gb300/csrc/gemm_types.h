// Parameters of the grouped GEMM kernels, and the host-side plan the layer
// composites use to launch the GEMM in parts (private to liboes).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "oes.h"

namespace oes {

struct GemmMaps {
  CUtensorMap a;   // 16-bit weights [S][rows][K] (bf16 path)
  CUtensorMap q;   // NVFP4 values [S][rows][K/2] bytes
  CUtensorMap sc;  // NVFP4 scales [S][K/64][rows] u32
  CUtensorMap b;   // GEMM2: h [cap][I]
};

struct GemmParams {
  const int32_t* sorted_ids;
  const int32_t* block_expert;
  const int32_t* n_post_pad;
  const int32_t* e2s;
  const uint8_t* flags;  // [E] group of each expert (filtered launches)
  const int32_t* gcount;  // [groups] experts in each group, or null
  int filter;            // 0 all blocks; g > 0 the blocks of experts with flags[e] == g
  int a4;                // W4A4: x and h hold NVFP4-quantised activations
  const float* act;      // W4A4: device [2] activation scales of GEMM1, GEMM2
  const uint8_t* pool;
  int64_t row_bytes;
  int64_t scal_off;  // NVFP4: byte offset of the fp32 scalars in a row
  int R, k, BN, H, I, E, S;
  int n_mtiles, n_kc, up_row0;  // up_row0: first up row of w13 (= I)
  int ks;          // K splits of a tile: 1, or 2 (GEMM1 of the weight-major kernel)
  float* part;     // ks = 2: fp32 gate and up sums of each half of each tile [tiles][2][2][BN][128]
  int32_t* tcount;  // ks = 2: halves finished per tile and epilogue warp [tiles][4], zero before GEMM1
  int NS, NR;                   // pipeline depths
  uint32_t tmem_cols;
  const uint16_t* xg;  // GEMM1: token rows to gather, [T, H] (bf16, or f16 for NVFP4)
  uint16_t* h;  // [cap, I]
  uint16_t* y;  // [R, H] bf16
  int32_t* status;
};

// Everything needed to launch GEMM1 / GEMM2 / combine of one call.
struct GemmPlan {
  GemmMaps m1, m2;
  GemmParams p1, p2;
  bool empty, tm;
  int split_tiles;  // > 0: GEMM1 splits K over this many tiles at most
  int32_t* counters;  // GEMM1's split counts
  int n_counters;
  int wf, a4, T, k, H, E;
  uint16_t* y;
  const uint16_t* x;        // the chunk's x (bf16)
  uint16_t* x16;            // its 16-bit copy for NVFP4 weights (workspace)
  float* act;               // W4A4 activation scales (workspace)
  const float *in13, *in2;  // W4A4: the layer's input scales
  int32_t* status;
};

// host only: validation, tensor maps, kernel parameters
int gemm_prepare(const oes_routed_experts* v, const uint16_t* x, int T, int k,
                 const int32_t* sorted_ids, const int32_t* block_expert, const int32_t* n_post_pad,
                 int B, void* workspace, size_t workspace_bytes, int32_t* status, GemmPlan* plan);
// the x kernels of a prepared GEMM (NVFP4 weights), on `stream`
int gemm_prepare_x(const GemmPlan& plan, cudaStream_t stream);
// The int32 words GEMM1's K split counts in, to be zeroed before the plan's
// first gemm_run (none when it does not split); a composite call has its
// align zero them.
struct GemmCounters {
  int32_t* ptr;
  int n;
};
inline GemmCounters gemm_counters(const GemmPlan& plan) {
  if (plan.empty || plan.n_counters <= 0) return {nullptr, 0};
  return {plan.counters, plan.n_counters};
}
// filter: 0 every block; g > 0 the blocks of experts with flags[e] == g
int gemm_run(const GemmPlan& plan, int filter, const uint8_t* flags, const int32_t* gcount,
             cudaStream_t stream);
int gemm_combine(const GemmPlan& plan, const int32_t* ids, const float* weights, uint16_t* out,
                 cudaStream_t stream);

}  // namespace oes
