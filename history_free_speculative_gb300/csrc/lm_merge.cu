// Deterministic merge of the LM-head records: for each row, the best
// (score, token id) over all vocabulary slabs (ties -> lowest id) and the
// log-sum-exp of logit/T, combined in a fixed order.
#include "internal.h"

namespace dlite {

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  const float mm = fmaxf(m, m2);
  s = s * expf(m - mm) + s2 * expf(m2 - mm);
  m = mm;
}

// One warp per row: merge the per-tile records in a fixed order.
__global__ void lm_merge_kernel(const LmRec* rec, int n_tiles, int rows, int K, float inv_T,
                                int32_t* cand, dlite_qstats* qs) {
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const bool sampling = inv_T > 0.f;
  LmRec best;
  best.best = -INFINITY;
  best.idx = 0x7fffffff;
  best.logit = 0.f;
  best.m = -INFINITY;
  best.s = 0.f;
  for (int tI = lane; tI < n_tiles; tI += 32) {
    const LmRec o = rec[(size_t)tI * rows + r];
    if (better(o.best, o.idx, best.best, best.idx)) {
      best.best = o.best; best.idx = o.idx; best.logit = o.logit;
    }
    if (sampling) lse_merge(best.m, best.s, o.m, o.s);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    LmRec other;
    other.best = __shfl_xor_sync(0xffffffffu, best.best, o);
    other.idx = __shfl_xor_sync(0xffffffffu, best.idx, o);
    other.logit = __shfl_xor_sync(0xffffffffu, best.logit, o);
    other.m = __shfl_xor_sync(0xffffffffu, best.m, o);
    other.s = __shfl_xor_sync(0xffffffffu, best.s, o);
    if (better(other.best, other.idx, best.best, best.idx)) {
      best.best = other.best; best.idx = other.idx; best.logit = other.logit;
    }
    if (sampling) lse_merge(best.m, best.s, other.m, other.s);
  }
  if (lane == 0) {
    cand[r] = best.idx;
    if (qs) {
      qs[r].logit = best.logit;
      qs[r].lse = sampling ? best.m + logf(best.s) : NAN;
    }
  }
}

cudaError_t launch_lm_merge(const LmRec* rec, int n_tiles, int rows, int K, float inv_T,
                            int32_t* cand, dlite_qstats* qs, cudaStream_t s) {
  const int wpb = 8;
  lm_merge_kernel<<<(rows + wpb - 1) / wpb, wpb * 32, 0, s>>>(rec, n_tiles, rows, K, inv_T, cand, qs);
  return cudaGetLastError();
}

}  // namespace dlite
