// LM-head merge and exact re-scoring.
//
// The tensor-core pass scores every vocabulary id with the bf16 rounding of
// the head state h and keeps, per row and vocabulary slab, the 4 best
// (score, id) plus the slab's log-sum-exp partials. This kernel merges those
// lists over all slabs in a fixed order (ties -> lowest id), then recomputes
// the logits of the 4 finalists exactly (fp32 h against the stored weights,
// fp32 accumulation) and decides among them. The bf16 rounding of h moves a
// logit by ~1e-3 (D = 4096, weights ~N(0, 0.02^2)), far less than the usual
// gap between the first and the fifth best score, so the re-scored winner is
// the winner of the exact product; rows where the fourth finalist is within
// kCloseCall of the first are counted as close calls.
#include "internal.h"

namespace dlite {

constexpr float kCloseCall = 0.02f;  // score units (logit, or logit/T when sampling)

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
  s = s * __expf(m - mm) + s2 * __expf(m2 - mm);
  m = mm;
}

// Merge two descending top-k lists into (sc, id).
__device__ __forceinline__ void topk_merge(float (&sc)[kTopK], int (&id)[kTopK],
                                           const float (&sc2)[kTopK], const int (&id2)[kTopK]) {
  float o[kTopK];
  int oi[kTopK];
  int a = 0, b = 0;  // a, b <= k at step k: every read below is in range
#pragma unroll
  for (int k = 0; k < kTopK; ++k) {
    const bool take_a = better(sc[a], id[a], sc2[b], id2[b]) || (sc[a] == sc2[b] && id[a] == id2[b]);
    if (take_a) {
      o[k] = sc[a];
      oi[k] = id[a];
      // drop an identical entry in the other list (the same id cannot appear twice)
      if (sc2[b] == sc[a] && id2[b] == id[a]) ++b;
      ++a;
    } else {
      o[k] = sc2[b];
      oi[k] = id2[b];
      ++b;
    }
  }
#pragma unroll
  for (int k = 0; k < kTopK; ++k) {
    sc[k] = o[k];
    id[k] = oi[k];
  }
}

__device__ __forceinline__ float exact_logit(const LmMergeArgs& a, int v, const float* h) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  if (a.Ef) {
    const float* e = a.Ef + (size_t)v * a.D;
    for (int d = lane * 4; d < a.D; d += 128) {
      const float4 ev = *reinterpret_cast<const float4*>(e + d);
      const float4 hv = *reinterpret_cast<const float4*>(h + d);
      acc = fmaf(ev.x, hv.x, fmaf(ev.y, hv.y, fmaf(ev.z, hv.z, fmaf(ev.w, hv.w, acc))));
    }
  } else {
    for (int d = lane * 4; d < a.D; d += 128) {
      const uint2 raw = *reinterpret_cast<const uint2*>(a.Eb + tiled_index(v, d, a.D));
      const __nv_bfloat162 e01 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
      const __nv_bfloat162 e23 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
      const float4 hv = *reinterpret_cast<const float4*>(h + d);
      acc = fmaf(__low2float(e01), hv.x, acc);
      acc = fmaf(__high2float(e01), hv.y, acc);
      acc = fmaf(__low2float(e23), hv.z, acc);
      acc = fmaf(__high2float(e23), hv.w, acc);
    }
  }
  return warp_sum(acc);
}

// One warp per row.
__global__ void lm_merge_kernel(const LmMergeArgs a) {
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= a.rows) return;
  const bool sampling = a.inv_T > 0.f;
  float sc[kTopK];
  int id[kTopK];
#pragma unroll
  for (int k = 0; k < kTopK; ++k) {
    sc[k] = -INFINITY;
    id[k] = 0x7fffffff;
  }
  float m = -INFINITY, s = 0.f;
  for (int t = lane; t < a.n_tiles; t += 32) {
    const LmRec rec = a.rec[(size_t)t * a.rows + r];
    topk_merge(sc, id, rec.sc, rec.id);
    if (sampling) lse_merge(m, s, rec.m, rec.s);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float sc2[kTopK];
    int id2[kTopK];
#pragma unroll
    for (int k = 0; k < kTopK; ++k) {
      sc2[k] = __shfl_xor_sync(0xffffffffu, sc[k], o);
      id2[k] = __shfl_xor_sync(0xffffffffu, id[k], o);
    }
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    topk_merge(sc, id, sc2, id2);
    if (sampling) lse_merge(m, s, m2, s2);
  }
  // exact re-scoring of the finalists
  const float* h = a.h + (size_t)r * a.D;
  uint32_t pos = 0, req = 0;
  if (sampling) {
    req = (uint32_t)(r / a.K);
    pos = (uint32_t)(a.pos[req] + (r % a.K) + 1);
  }
  float best = -INFINITY, blogit = 0.f;
  int bid = 0x7fffffff;
#pragma unroll
  for (int k = 0; k < kTopK; ++k) {
    const int v = id[k];
    if (v < 0 || v >= a.V) continue;  // fewer than kTopK ids (tiny vocabularies)
    const float l = exact_logit(a, v, h);
    float x = l;
    if (sampling) {
      const uint4 w = philox((uint32_t)v >> 2, pos, req, kTagGumbel, a.k0, a.k1);
      const uint32_t wx[4] = {w.x, w.y, w.z, w.w};
      x = l * a.inv_T + gumbel_from_bits(wx[v & 3]);
    }
    if (better(x, v, best, bid)) {
      best = x;
      bid = v;
      blogit = l;
    }
  }
  if (lane == 0) {
    a.cand[r] = bid;
    if (a.qs) {
      a.qs[r].logit = blogit;
      a.qs[r].lse = sampling ? m + logf(s) : NAN;
    }
    if (a.counters && sc[kTopK - 1] > sc[0] - kCloseCall) atomicAdd(a.counters + 4, 1ull);
  }
}

cudaError_t launch_lm_merge(const LmMergeArgs& a, cudaStream_t s) {
  const int wpb = 8;
  lm_merge_kernel<<<(a.rows + wpb - 1) / wpb, wpb * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dlite
