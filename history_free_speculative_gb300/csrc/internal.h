// Internal declarations shared by the DLite CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dlite.h"
#include "common.cuh"

#include <utility>

namespace dlite {

// Launch with programmatic stream serialization (see pdl_trigger / pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// LM-head record of a set of vocabulary columns for one row: the 4 best
// (score, id) in descending order (greedy: logit; sampling: the base-2
// Gumbel-max score logit log2(e)/T - log2(-log2 u)), from the bf16 product,
// and the LSE partials of those columns in base 2.
constexpr int kTopK = 4;
struct LmRec {
  float sc[kTopK];
  int id[kTopK];
  float m;  // max of logit log2(e) / T over the columns (sampling)
  float s;  // sum of 2^(logit log2(e) / T - m) over the columns (sampling)
};

// Merge of the LM-head records and exact re-scoring of the finalists.
struct LmMergeArgs {
  const LmRec* rec = nullptr;  // [n_tiles][rows]
  int n_tiles = 0, rows = 0, K = 0, D = 0, V = 0;
  float inv_T = 0.f;           // 0 = greedy
  double T = 0.0;              // the temperature (float32 value) for the re-scoring
  uint32_t k0 = 0, k1 = 0;
  const int64_t* pos = nullptr;
  const float* h = nullptr;    // [rows, D] fp32 head states
  const bf16* Eb = nullptr;    // exact LM weights (bf16, tiled layout) ...
  const float* Ef = nullptr;   // ... or fp32
  int32_t* cand = nullptr;
  dlite_qstats* qs = nullptr;
  unsigned long long* counters = nullptr;  // [4] = finalist sets that were close calls
};

cudaError_t launch_lm_merge(const LmMergeArgs& a, cudaStream_t s);

}  // namespace dlite
