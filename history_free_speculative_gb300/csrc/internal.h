// Internal declarations shared by the DLite CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "../../include/dlite.h"
#include "common.cuh"

namespace dlite {

// An operand of a tensor-core product: one or two bf16 planes (x ~ hi + lo),
// row-major [rows, ld].
struct Planes {
  const bf16* p[2] = {nullptr, nullptr};
  int n = 0;
  int ld = 0;
};

// GEMM: part[z][r][o] = sum over the k-range of split z of X[r, k] * W[o, k].
// Plane products: X0*W0, + X1*W0 when X has two planes, + X0*W1 when W has two.
struct GemmArgs {
  Planes X, W;
  int rows = 0, outs = 0, K = 0;
  int splits = 1;
  float* part = nullptr;  // [splits][rows][outs]
};

// LM-head records: the best (score, id) and the LSE partials of one vocabulary
// tile for one row.
struct LmRec {
  float best;   // best score (greedy: logit; sampling: logit/T + Gumbel)
  int idx;      // its token id
  float logit;  // the logit of that token
  float m;      // max of logit/T over the tile (sampling)
  float s;      // sum of exp(logit/T - m) over the tile (sampling)
};

struct LmArgs {
  Planes H;                // [rows, D]
  Planes E;                // [V, D]
  int rows = 0, V = 0, D = 0, K = 0;
  float inv_T = 0.f;       // 0 = greedy
  uint32_t k0 = 0, k1 = 0; // Philox key (seed)
  const int64_t* pos = nullptr;
  LmRec* rec = nullptr;    // [n_tiles][rows]
  int* status = nullptr;
};

int gemm_splits(int rows, int outs, int K);
size_t gemm_part_elems(int rows, int outs, int K);
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s);

int lm_tiles(int V);
cudaError_t launch_lm_head(const LmArgs& a, cudaStream_t s);
cudaError_t launch_lm_merge(const LmRec* rec, int n_tiles, int rows, int K, float inv_T,
                            int32_t* cand, dlite_qstats* qs, cudaStream_t s);

}  // namespace dlite
