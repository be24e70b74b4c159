// Internal declarations shared by the DLite CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dlite.h"
#include "common.cuh"

namespace dlite {

// LM-head record: the best (score, id) and the LSE partials of one vocabulary
// slab for one row.
struct LmRec {
  float best;   // best score (greedy: logit; sampling: logit/T + Gumbel)
  int idx;      // its token id
  float logit;  // the logit of that token
  float m;      // max of logit/T over the slab (sampling)
  float s;      // sum of exp(logit/T - m) over the slab (sampling)
};

cudaError_t launch_lm_merge(const LmRec* rec, int n_tiles, int rows, int K, float inv_T,
                            int32_t* cand, dlite_qstats* qs, cudaStream_t s);

}  // namespace dlite
