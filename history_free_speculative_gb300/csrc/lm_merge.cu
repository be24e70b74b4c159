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
//
// Sampling records are in base-2 units (score = logit log2(e) / T minus
// log2(-log2 u), an increasing map of the Gumbel-max score; LSE partials
// m = max logit log2(e) / T, s = sum 2^(. - m)); the finalists are re-scored
// in natural units, logit / T - log(-log u), and the LSE is returned in
// natural units.
#include "internal.h"

namespace dlite {

constexpr float kCloseCall = 0.02f;  // natural score units (logit, or logit/T when sampling)
constexpr float kLog2eM = 1.4426950408889634f;
constexpr float kLn2M = 0.6931471805599453f;

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
  s = s * exp2f(m - mm) + s2 * exp2f(m2 - mm);
  m = mm;
}

// Insert (x, v) into a descending top-k list held in registers (constant indices only).
__device__ __forceinline__ void cswap(float (&sc)[kTopK], int (&id)[kTopK], int k) {
  if (better(sc[k + 1], id[k + 1], sc[k], id[k])) {
    const float ts = sc[k];
    const int ti = id[k];
    sc[k] = sc[k + 1];
    id[k] = id[k + 1];
    sc[k + 1] = ts;
    id[k + 1] = ti;
  }
}
__device__ __forceinline__ void topk_insert(float (&sc)[kTopK], int (&id)[kTopK], float x, int v) {
  if (!better(x, v, sc[kTopK - 1], id[kTopK - 1])) return;
  sc[kTopK - 1] = x;
  id[kTopK - 1] = v;
#pragma unroll
  for (int k = kTopK - 2; k >= 0; --k) cswap(sc, id, k);
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
#pragma unroll 8
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

// One CTA of kMergeWarps warps per row: every thread folds a strided subset of the records
// into a register top-k + LSE, the warps combine by butterfly, thread 0
// combines the warps in a fixed order, and warps 0-3 re-score the 4 finalists
// exactly in parallel.

// Gumbel noise -log(-log u) of the uniform u01f(x) with full relative accuracy
// where it matters: for u within 2^-8 of 1, -log u is formed from the exact
// complement w = 1 - u by its series w + w^2/2 + w^3/3 (truncation < w^4/4,
// relative < 2^-26); elsewhere from the library logf.
__device__ __forceinline__ float gumbel_f(uint32_t x) {
  const uint32_t k = x >> 9;
  const float w = fmaf((float)(0x7fffffu - k), 1.1920928955078125e-07f, 5.9604644775390625e-08f);
  const float nl = w < 0.00390625f ? w * fmaf(w, fmaf(w, 1.f / 3.f, 0.5f), 1.f) : -logf(1.f - w);
  return -logf(nl);
}

template <int kMergeWarps>
__global__ void __launch_bounds__(kMergeWarps * 32) lm_merge_kernel(const LmMergeArgs a) {
  static_assert(kMergeWarps >= kTopK, "one warp per finalist");
  pdl_trigger();
  pdl_wait();
  __shared__ float wsc[kMergeWarps][kTopK];
  __shared__ int wid[kMergeWarps][kTopK];
  __shared__ float wm[kMergeWarps], wsum[kMergeWarps];
  __shared__ double fin_sc[kTopK];
  __shared__ float fin_logit[kTopK];
  __shared__ int fin_id[kTopK];
  __shared__ float row_m, row_s, row_sc0, row_sc3;
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool sampling = a.inv_T > 0.f;
  float sc[kTopK];
  int id[kTopK];
#pragma unroll
  for (int k = 0; k < kTopK; ++k) {
    sc[k] = -INFINITY;
    id[k] = 0x7fffffff;
  }
  float m = -INFINITY, s = 0.f;
  constexpr int kBatch = 4;  // records loaded before any is folded
  for (int t0 = threadIdx.x; t0 < a.n_tiles; t0 += blockDim.x * kBatch) {
    LmRec rec[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int t = t0 + u * blockDim.x;
      if (t < a.n_tiles) rec[u] = a.rec[(size_t)t * a.rows + r];
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (t0 + u * (int)blockDim.x >= a.n_tiles) break;
#pragma unroll
      for (int k = 0; k < kTopK; ++k) topk_insert(sc, id, rec[u].sc[k], rec[u].id[k]);
      if (sampling) lse_merge(m, s, rec[u].m, rec[u].s);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {  // both partners end with the same list (disjoint sets)
    float sc2[kTopK];
    int id2[kTopK];
#pragma unroll
    for (int k = 0; k < kTopK; ++k) {
      sc2[k] = __shfl_xor_sync(0xffffffffu, sc[k], o);
      id2[k] = __shfl_xor_sync(0xffffffffu, id[k], o);
    }
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
#pragma unroll
    for (int k = 0; k < kTopK; ++k) topk_insert(sc, id, sc2[k], id2[k]);
    if (sampling) lse_merge(m, s, m2, s2);
  }
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < kTopK; ++k) {
      wsc[warp][k] = sc[k];
      wid[warp][k] = id[k];
    }
    wm[warp] = m;
    wsum[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kMergeWarps; ++w) {
#pragma unroll
      for (int k = 0; k < kTopK; ++k) topk_insert(sc, id, wsc[w][k], wid[w][k]);
      if (sampling) lse_merge(m, s, wm[w], wsum[w]);
    }
#pragma unroll
    for (int k = 0; k < kTopK; ++k) fin_id[k] = id[k];
    row_m = m;
    row_s = s;
    row_sc0 = sc[0];
    row_sc3 = sc[kTopK - 1];
  }
  __syncthreads();
  // exact re-scoring: warp k < kTopK takes finalist k
  const float* h = a.h + (size_t)r * a.D;
  if (warp < kTopK) {
    const int v = fin_id[warp];
    double x = -INFINITY;
    float l = 0.f;
    if (v >= 0 && v < a.V) {  // fewer than kTopK ids on tiny vocabularies
      l = exact_logit(a, v, h);
      x = l;
      if (sampling) {
        const uint32_t req = (uint32_t)(r / a.K);
        const uint32_t pos = (uint32_t)(a.pos[req] + (r % a.K) + 1);
        const uint4 w = philox((uint32_t)v >> 2, pos, req, kTagGumbel, a.k0, a.k1);
        const uint32_t wx[4] = {w.x, w.y, w.z, w.w};
        x = (double)l / a.T + (double)gumbel_f(wx[v & 3]);
      }
    }
    if (lane == 0) {
      fin_sc[warp] = x;
      fin_logit[warp] = l;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double best = -INFINITY;
    float blogit = 0.f;
    int bid = 0x7fffffff;
    for (int k = 0; k < kTopK; ++k) {
      const int v = fin_id[k];
      if (v < 0 || v >= a.V) continue;
      if (fin_sc[k] > best || (fin_sc[k] == best && v < bid)) {
        best = fin_sc[k];
        bid = v;
        blogit = fin_logit[k];
      }
    }
    a.cand[r] = bid;
    if (a.qs) {
      a.qs[r].logit = blogit;
      a.qs[r].lse = sampling ? (row_m + log2f(row_s)) * kLn2M : NAN;
    }
    const float band = sampling ? kCloseCall * kLog2eM : kCloseCall;
    if (a.counters && row_sc3 > row_sc0 - band) atomicAdd(a.counters + 4, 1ull);
  }
}

cudaError_t launch_lm_merge(const LmMergeArgs& a, cudaStream_t s) {
  return launch_pdl(lm_merge_kernel<4>, dim3(a.rows), dim3(4 * 32), 0, s, a);
}

}  // namespace dlite
