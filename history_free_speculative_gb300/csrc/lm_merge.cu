// LM-head merge and exact re-scoring.
//
// The tensor-core pass scores the vocabulary with the bf16 rounding of the
// head state h and keeps, per row and vocabulary walk, the 4 best
// (score, id) plus the log-sum-exp partials. This kernel merges those lists
// over all walks in a fixed order (ties -> lowest id), then decides among the
// finalists with exact logits (fp32 h against the stored weights, fp32
// accumulation). The bf16 rounding of h moves a logit by ~1e-3 (D = 4096,
// weights ~N(0, 0.02^2)), far less than the usual gap between the first and
// the fifth best score, so the exact decision is the decision of the exact
// product.
// Greedy: the entries are vocabulary ids; the 4 finalists are re-scored and
// the best taken (rows whose fourth finalist is within kCloseCall of the first
// are counted as close calls).
// Sampling (the two-level draw): the entries are 16-id chunks scored in base-2
// units (see the fold in tc_device.cuh); every finalist chunk within
// kChunkBand of the best is re-scored exactly (16 logits each), the chunk
// with the best exact score L_k - log(-log u_k) is chosen, and the draft token
// is the inverse CDF of exp(l_v / T - L_k) inside it at the uniform of
// Philox(k, position, request, tag 8) word 0 (rows with more than one chunk in
// the band are counted as close calls). The LSE is returned in natural units.
#include "internal.h"

namespace dlite {

constexpr float kCloseCall = 0.02f;  // natural score units (logit, or logit/T when sampling)
// finalist chunks within this many natural units of the best approximate
// chunk score are re-scored exactly (> 10x the score error of bf16 h)
constexpr float kChunkBand = 0.05f;
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

// Partial exact logit of id v over columns [lo, hi) (fp32 accumulation; the
// warp's lanes take 4 columns each per 128, all loads issued before use).
template <int kU>
__device__ __forceinline__ float exact_logit_part(const LmMergeArgs& a, int v, const float* h, int lo, int hi) {
  const int lane = threadIdx.x & 31;
  float acc0 = 0.f, acc1 = 0.f;
  for (int d0 = lo + lane * 4; d0 < hi; d0 += 128 * kU) {
    float4 ev[kU], hv[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int d = d0 + 128 * u;
      if (d < hi) {
        hv[u] = *reinterpret_cast<const float4*>(h + d);
        if (a.Ef) {
          ev[u] = *reinterpret_cast<const float4*>(a.Ef + (size_t)v * a.D + d);
        } else {
          const uint2 raw = *reinterpret_cast<const uint2*>(a.Eb + tiled_index(v, d, a.D));
          const __nv_bfloat162 e01 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
          const __nv_bfloat162 e23 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
          ev[u] = make_float4(__low2float(e01), __high2float(e01), __low2float(e23), __high2float(e23));
        }
      } else {
        hv[u] = ev[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; u += 2) {
      acc0 = fmaf(ev[u].x, hv[u].x, fmaf(ev[u].y, hv[u].y, fmaf(ev[u].z, hv[u].z, fmaf(ev[u].w, hv[u].w, acc0))));
      acc1 = fmaf(ev[u + 1].x, hv[u + 1].x,
                  fmaf(ev[u + 1].y, hv[u + 1].y, fmaf(ev[u + 1].z, hv[u + 1].z, fmaf(ev[u + 1].w, hv[u + 1].w, acc1))));
    }
  }
  return warp_sum(acc0 + acc1);
}

// The 4 best (score, id) over the lanes' descending lists by a tournament:
// four warp-wide arg-max reductions, the owner of each winner popping it.
// Every lane returns the same list; the lanes' lists are consumed.
__device__ __forceinline__ void warp_top4(float (&sc)[kTopK], int (&id)[kTopK], float (&osc)[kTopK],
                                          int (&oid)[kTopK]) {
#pragma unroll
  for (int k = 0; k < kTopK; ++k) {
    float bv = sc[0];
    int bi = id[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(v2, i2, bv, bi)) {
        bv = v2;
        bi = i2;
      }
    }
    osc[k] = bv;
    oid[k] = bi;
    if (id[0] == bi && sc[0] == bv) {  // ids are unique, except the empty entries
#pragma unroll
      for (int j = 0; j + 1 < kTopK; ++j) {
        sc[j] = sc[j + 1];
        id[j] = id[j + 1];
      }
      sc[kTopK - 1] = -INFINITY;
      id[kTopK - 1] = 0x7fffffff;
    }
  }
}

// The 16 exact logits of chunk k, this warp's share: lane L of warp w takes the
// column quads d = 4 (L + 32 (w + nw i)), i = 0, 1, ..., for 8 ids at a time
// (the 8 rows' loads of a quad in flight together), then the lanes' sums are
// reduced; returns this warp's partial for id t in lane t (t < 16).
__device__ __forceinline__ float chunk_logits_part(const LmMergeArgs& a, int k, const float* h, int nw) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kIds = kChunk / 2;
  const int v0 = k * kChunk;
  const int nv = min(kChunk, a.V - v0);
  const int stride = 4 * 32 * nw;
  float mine = 0.f;
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    float acc[kIds];
#pragma unroll
    for (int t = 0; t < kIds; ++t) acc[t] = 0.f;
    if (!a.Ef) {
      // bf16 weights: up to four quads per id in flight, kept as raw bf16 pairs
      // (32 x 8 bytes per lane) until the arithmetic, one round trip per half
      // at D <= 4096
      for (int d0 = 4 * (lane + 32 * warp); d0 < a.D; d0 += 4 * stride) {
        uint2 raw[4][kIds];
        float4 hv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int d = d0 + u * stride;
          hv[u] = d < a.D ? *reinterpret_cast<const float4*>(h + d) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int t = 0; t < kIds; ++t)
            raw[u][t] = d < a.D && half * kIds + t < nv
                            ? *reinterpret_cast<const uint2*>(a.Eb + tiled_index(v0 + half * kIds + t, d, a.D))
                            : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int t = 0; t < kIds; ++t) {
            const float4 e = make_float4(__uint_as_float(raw[u][t].x << 16), __uint_as_float(raw[u][t].x & 0xffff0000u),
                                         __uint_as_float(raw[u][t].y << 16), __uint_as_float(raw[u][t].y & 0xffff0000u));
            acc[t] = fmaf(e.x, hv[u].x, fmaf(e.y, hv[u].y, fmaf(e.z, hv[u].z, fmaf(e.w, hv[u].w, acc[t]))));
          }
      }
    } else {
      for (int d = 4 * (lane + 32 * warp); d < a.D; d += stride) {
        const float4 hv = *reinterpret_cast<const float4*>(h + d);
        float4 ev[kIds];
#pragma unroll
        for (int t = 0; t < kIds; ++t)
          ev[t] = half * kIds + t < nv
                      ? *reinterpret_cast<const float4*>(a.Ef + (size_t)(v0 + half * kIds + t) * a.D + d)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int t = 0; t < kIds; ++t)
          acc[t] = fmaf(ev[t].x, hv.x, fmaf(ev[t].y, hv.y, fmaf(ev[t].z, hv.z, fmaf(ev[t].w, hv.w, acc[t]))));
      }
    }
#pragma unroll
    for (int t = 0; t < kIds; ++t) {
      const float v = warp_sum(acc[t]);
      if (lane == half * kIds + t) mine = v;
    }
  }
  return mine;
}

// Short rows (D <= 512, the gated head's W_o product): the exact logits of
// every finalist chunk in the band at once, into chunk_l[j][t]. The n_band x 16
// ids are dealt to the warps round-robin, four ids of a warp at a time with all
// their loads in flight (one round trip for the usual one or two chunks,
// instead of one per chunk and half-chunk); lanes take 4-column quads.
__device__ __forceinline__ void band_logits_short(const LmMergeArgs& a, const int* fin, int n_band, const float* h,
                                                  float (*chunk_l)[kChunk], int nw) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float4 hv[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int d = 4 * lane + 128 * u;
    hv[u] = d < a.D ? *reinterpret_cast<const float4*>(h + d) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int n_ids = n_band * kChunk;
  for (int i0 = warp; i0 < n_ids; i0 += 4 * nw) {
    float acc[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      acc[t] = 0.f;
      const int ii = i0 + t * nw, j = ii / kChunk, tt = ii % kChunk;
      const int v = (ii < n_ids ? fin[j] : 0) * kChunk + tt;
      if (ii >= n_ids || v >= a.V) continue;
      float4 ev[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int d = 4 * lane + 128 * u;
        ev[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (d < a.D) {
          if (a.Ef) {
            ev[u] = *reinterpret_cast<const float4*>(a.Ef + (size_t)v * a.D + d);
          } else {
            const uint2 raw = *reinterpret_cast<const uint2*>(a.Eb + tiled_index(v, d, a.D));
            const __nv_bfloat162 e01 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
            const __nv_bfloat162 e23 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
            ev[u] = make_float4(__low2float(e01), __high2float(e01), __low2float(e23), __high2float(e23));
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        acc[t] = fmaf(ev[u].x, hv[u].x, fmaf(ev[u].y, hv[u].y, fmaf(ev[u].z, hv[u].z, fmaf(ev[u].w, hv[u].w, acc[t]))));
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int ii = i0 + t * nw;
      const float sum = warp_sum(acc[t]);
      if (lane == 0 && ii < n_ids) chunk_l[ii / kChunk][ii % kChunk] = sum;
    }
  }
}

__device__ __forceinline__ void warp_lse(float& m, float& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {  // both partners form the same two terms
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, m2, s2);
  }
}

// One CTA of kMergeWarps warps per row: each thread takes the records
// t = tid, tid + blockDim, ... (normally one: its record's list is already
// sorted), each warp reduces its lanes' lists by tournament, warp 0 reduces
// the warps' lists the same way, and the warps re-score the 4 finalists
// exactly, two warps (half of the columns each) per finalist.

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

// kSampling: the sampling form (<= 128 registers: two CTAs per SM, as many rows
// as there are; no early launch of the successor: the sampling verification's
// CTAs waiting on these SMs slowed this kernel by about 2x, and so did the
// gated head's next step with the vocabulary stream behind it); the greedy
// form (few rows in practice; deeper loads for the finalists, the successor
// may launch early).
template <int kMergeWarps, bool kSampling>
__global__ void __launch_bounds__(kMergeWarps * 32, kSampling ? 2 : 1) lm_merge_kernel(const LmMergeArgs a) {
  static_assert(kMergeWarps == 2 * kTopK, "two warps per finalist");
  if (!kSampling) pdl_trigger();
  pdl_wait();
  __shared__ float wsc[kMergeWarps][kTopK];
  __shared__ int wid[kMergeWarps][kTopK];
  __shared__ float wm[kMergeWarps], wsum[kMergeWarps];
  __shared__ float part[kMergeWarps];
  __shared__ int fin_id[kTopK];
  __shared__ float row_m, row_s, row_sc0, row_sc3;
  __shared__ float chunk_l[kTopK][kChunk];  // sampling: exact logits of the finalist chunks
  __shared__ float chunk_part[kMergeWarps][kChunk];
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr bool sampling = kSampling;
  float sc[kTopK];
  int id[kTopK];
#pragma unroll
  for (int k = 0; k < kTopK; ++k) {
    sc[k] = -INFINITY;
    id[k] = 0x7fffffff;
  }
  float m = -INFINITY, s = 0.f;
  if ((int)threadIdx.x < a.n_tiles) {  // the first record is this lane's list as it stands
    const LmRec rec = a.rec[(size_t)threadIdx.x * a.rows + r];
#pragma unroll
    for (int k = 0; k < kTopK; ++k) {
      sc[k] = rec.sc[k];
      id[k] = rec.id[k];
    }
    m = rec.m;
    s = rec.s;
  }
  for (int t = threadIdx.x + blockDim.x; t < a.n_tiles; t += blockDim.x) {
    const LmRec rec = a.rec[(size_t)t * a.rows + r];
#pragma unroll
    for (int k = 0; k < kTopK; ++k) topk_insert(sc, id, rec.sc[k], rec.id[k]);
    if (sampling) lse_merge(m, s, rec.m, rec.s);
  }
  float osc[kTopK];
  int oid[kTopK];
  warp_top4(sc, id, osc, oid);
  if (sampling) warp_lse(m, s);
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < kTopK; ++k) {
      wsc[warp][k] = osc[k];
      wid[warp][k] = oid[k];
    }
    wm[warp] = m;
    wsum[warp] = s;
  }
  __syncthreads();
  if (warp == 0) {  // the same reduction over the warps' lists, lane w holding warp w's
#pragma unroll
    for (int k = 0; k < kTopK; ++k) {
      sc[k] = lane < kMergeWarps ? wsc[lane][k] : -INFINITY;
      id[k] = lane < kMergeWarps ? wid[lane][k] : 0x7fffffff;
    }
    m = lane < kMergeWarps ? wm[lane] : -INFINITY;
    s = lane < kMergeWarps ? wsum[lane] : 0.f;
    warp_top4(sc, id, osc, oid);
    if (sampling) warp_lse(m, s);
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < kTopK; ++k) {
        fin_id[k] = oid[k];
        wsc[0][k] = osc[k];  // the finalists' approximate scores (warp 0's list slot is free now)
      }
      row_m = m;
      row_s = s;
      row_sc0 = osc[0];
      row_sc3 = osc[kTopK - 1];
    }
  }
  __syncthreads();
  const float* h = a.h + (size_t)r * a.D;
  if constexpr (kSampling) {
    // exact logits of the finalist chunks in the band (a prefix of the sorted
    // finalists): short rows all at once; otherwise chunk by chunk, every warp
    // taking a slice of the columns of all 16 ids, the warps' partials added in
    // warp order
    int n_band = 0;
    while (n_band < kTopK && fin_id[n_band] >= 0 && (long long)fin_id[n_band] * kChunk < a.V &&
           wsc[0][n_band] >= row_sc0 - kChunkBand * kLog2eM)
      ++n_band;
    if (a.D <= 512) {
      band_logits_short(a, fin_id, n_band, h, chunk_l, kMergeWarps);
      __syncthreads();
    }
    for (int j = 0; j < (a.D <= 512 ? 0 : n_band); ++j) {
      const int k = fin_id[j];
      const float pv = chunk_logits_part(a, k, h, kMergeWarps);
      if (lane < kChunk) chunk_part[warp][lane] = pv;
      __syncthreads();
      if (warp == 0 && lane < kChunk) {
        float l = 0.f;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) l += chunk_part[w][lane];
        chunk_l[j][lane] = l;
      }
      __syncthreads();
    }
    if (warp == 0) {
      // lane j: the exact score of finalist chunk j; the best by a 4-lane
      // reduction (ties -> lowest chunk id). fp32 with the accurate library
      // exp / log (this GPU's float64 units are far too slow for a per-row
      // tail): the decisions match the float64 oracle except where a score
      // or a CDF step is within ~1e-6 of the deciding value.
      const uint32_t req = (uint32_t)(r / a.K);
      const uint32_t pos = (uint32_t)(a.pos[req] + (r % a.K) + 1);
      const float invT = 1.f / (float)a.T;
      float x = -INFINITY;
      int kk = 0x7fffffff, n_in = 0;
      if (lane < kTopK) {
        const int kc = fin_id[lane];
        if (kc >= 0 && (long long)kc * kChunk < a.V && wsc[0][lane] >= row_sc0 - kChunkBand * kLog2eM) {
          const int nv = min(kChunk, a.V - kc * kChunk);
          float mx = -INFINITY, tot = 0.f;
          for (int t = 0; t < nv; ++t) mx = fmaxf(mx, chunk_l[lane][t] * invT);
          for (int t = 0; t < nv; ++t) tot += expf(chunk_l[lane][t] * invT - mx);
          const uint4 w = philox((uint32_t)kc >> 2, pos, req, kTagGumbel, a.k0, a.k1);
          const uint32_t wx[4] = {w.x, w.y, w.z, w.w};
          x = mx + logf(tot) + gumbel_f(wx[kc & 3]);
          kk = kc;
          n_in = 1;
        }
      }
#pragma unroll
      for (int o = 1; o < kTopK; o <<= 1) {
        const float x2 = __shfl_xor_sync(0xffffffffu, x, o);
        const int k2 = __shfl_xor_sync(0xffffffffu, kk, o);
        if (x2 > x || (x2 == x && k2 < kk)) {
          x = x2;
          kk = k2;
        }
      }
      n_in += __shfl_xor_sync(0xffffffffu, n_in, 1);
      n_in += __shfl_xor_sync(0xffffffffu, n_in, 2);
      if (lane == 0 && kk == 0x7fffffff) {  // no finalist (cannot happen with V >= 1): id 0
        a.cand[r] = 0;
        if (a.qs) a.qs[r].logit = 0.f;
      } else if (lane == 0) {
        int jw = 0;  // the finalist slot of the chosen chunk
        for (int t = 0; t < kTopK; ++t)
          if (fin_id[t] == kk) jw = t;
        const int nv = min(kChunk, a.V - kk * kChunk);
        float m2 = -INFINITY, t2 = 0.f;
        for (int t = 0; t < nv; ++t) m2 = fmaxf(m2, chunk_l[jw][t] * invT);
        for (int t = 0; t < nv; ++t) t2 += expf(chunk_l[jw][t] * invT - m2);
        const float th = u01f(philox((uint32_t)kk, pos, req, kTagPick, a.k0, a.k1).x) * t2;
        float c = 0.f;
        int pick = nv - 1;  // the smallest id whose running sum passes the threshold
        for (int t = 0; t + 1 < nv; ++t) {
          c += expf(chunk_l[jw][t] * invT - m2);
          if (c > th) {
            pick = t;
            break;
          }
        }
        a.cand[r] = kk * kChunk + pick;
        if (a.qs) {
          a.qs[r].logit = chunk_l[jw][pick];
          a.qs[r].lse = (row_m + log2f(row_s)) * kLn2M;
        }
        if (a.counters && n_in > 1) atomicAdd(a.counters + 4, 1ull);
      }
    }
    return;
  }
  // greedy: exact re-scoring, warps 2k and 2k + 1 take the two halves of finalist k
  {
    const int v = fin_id[warp >> 1];
    const int half = (a.D / 2 + 3) & ~3;
    const int lo = (warp & 1) ? half : 0, hi = (warp & 1) ? a.D : half;
    float p = 0.f;
    if (v >= 0 && v < a.V) p = exact_logit_part<16>(a, v, h, lo, hi);  // fewer than kTopK ids on tiny vocabularies
    if (lane == 0) part[warp] = p;
  }
  __syncthreads();
  if (warp == 0) {  // lane k scores finalist k; the best by a 4-lane reduction (ties -> lowest id)
    float x = -INFINITY;
    int v = 0x7fffffff;
    if (lane < kTopK) {
      const int fv = fin_id[lane];
      if (fv >= 0 && fv < a.V) {
        v = fv;
        x = part[2 * lane] + part[2 * lane + 1];
      }
    }
    float l = x;
#pragma unroll
    for (int o = 1; o < kTopK; o <<= 1) {
      const float x2 = __shfl_xor_sync(0xffffffffu, x, o);
      const int v2 = __shfl_xor_sync(0xffffffffu, v, o);
      if (x2 > x || (x2 == x && v2 < v)) {
        x = x2;
        v = v2;
      }
    }
    l = x;
    if (lane == 0) {
      a.cand[r] = v;
      if (a.qs) {
        a.qs[r].logit = l;
        a.qs[r].lse = NAN;
      }
      if (a.counters && row_sc3 > row_sc0 - kCloseCall) atomicAdd(a.counters + 4, 1ull);
    }
  }
}

cudaError_t launch_lm_merge(const LmMergeArgs& a, cudaStream_t s) {
  if (a.inv_T > 0.f) return launch_pdl(lm_merge_kernel<2 * kTopK, true>, dim3(a.rows), dim3(2 * kTopK * 32), 0, s, a);
  return launch_pdl(lm_merge_kernel<2 * kTopK, false>, dim3(a.rows), dim3(2 * kTopK * 32), 0, s, a);
}

}  // namespace dlite
