// DLite round kernels other than the tensor-core products: staging, block
// attention (with the QKV split-K reduction and RoPE fused in), residual +
// RMSNorm epilogues, SwiGLU, the sequential head's serial chain, and the
// verify / commit kernels.
#include "kernels.h"

namespace dlite {

// ---------------------------------------------------------------- helpers

template <typename T>
__device__ __forceinline__ float ld_elem(const void* p, size_t i) {
  return to_f32(reinterpret_cast<const T*>(p)[i]);
}

__device__ __forceinline__ void store_planes(bf16* const* pl, int n, size_t i, float v) {
  if (n == 2) {
    bf16 hi, lo;
    split_bf16(v, hi, lo);
    pl[0][i] = hi;
    pl[1][i] = lo;
  } else {
    pl[0][i] = __float2bfloat16_rn(v);
  }
}

constexpr int kRowThreads = 512;  // two or more CTAs per SM (rows in one wave)
constexpr int kRowVec = 8;        // float4 chunks per thread at most (D <= 16384)

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"((uint32_t)__cvta_generic_to_shared(local)), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ float4 f4add(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

template <int kDepth = 4>
__device__ __forceinline__ float4 sum_splits4(const float* base, size_t stride, int S) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < S; s += kDepth) {  // up to kDepth loads in flight, added in plane order
    float4 t[kDepth];
#pragma unroll
    for (int k = 0; k < kDepth; ++k)
      if (s + k < S) t[k] = *reinterpret_cast<const float4*>(base + (size_t)(s + k) * stride);
#pragma unroll
    for (int k = 0; k < kDepth; ++k)
      if (s + k < S) acc = f4add(acc, t[k]);
  }
  return acc;
}

// One float4 of a split-K product: its first plane, the plane stride, the planes.
struct SplitSrc {
  const float* p = nullptr;
  size_t stride = 0;
  int n = 0;
};
// Two such sums at once: up to kDepth loads of each in flight together, each
// sum added in plane order from zero (the same result as sum_splits4).
template <int kDepth>
__device__ __forceinline__ void sum_splits4x2(const SplitSrc& s0, const SplitSrc& s1, float4& r0, float4& r1) {
  r0 = make_float4(0.f, 0.f, 0.f, 0.f);
  r1 = r0;
  const int nmax = s0.n > s1.n ? s0.n : s1.n;
  for (int s = 0; s < nmax; s += kDepth) {
    float4 t0[kDepth], t1[kDepth];
#pragma unroll
    for (int k = 0; k < kDepth; ++k) {
      if (s + k < s0.n) t0[k] = *reinterpret_cast<const float4*>(s0.p + (size_t)(s + k) * s0.stride);
      if (s + k < s1.n) t1[k] = *reinterpret_cast<const float4*>(s1.p + (size_t)(s + k) * s1.stride);
    }
#pragma unroll
    for (int k = 0; k < kDepth; ++k) {
      if (s + k < s0.n) r0 = f4add(r0, t0[k]);
      if (s + k < s1.n) r1 = f4add(r1, t1[k]);
    }
  }
}

__device__ __forceinline__ void store4_planes(bf16* const* pl, int n, size_t i, float4 v) {
  store_planes(pl, n, i, v.x);
  store_planes(pl, n, i + 1, v.y);
  store_planes(pl, n, i + 2, v.z);
  store_planes(pl, n, i + 3, v.w);
}

// ---------------------------------------------------------------- K1: staging
// Rows [0, B*m): z_{b,j} = RMSNorm(hidden_{b,j} + e_depth_j) * g_stage.
// Rows [B*m, B*m + B*(K+1)): local rows x_{b,0} = E[anchor_b], x_{b,i} = e_ph,
// and y = RMSNorm(x) * g_attn (layer 0 input of the QKV product).
// One CTA of 1024 threads per row, 4 consecutive elements per thread and step.
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const bf16* p) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
  return make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
}

template <typename T, int kVec>  // kVec: float4 chunks of a row per thread at most
__global__ void __launch_bounds__(1024) stage_kernel(StageArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int row = blockIdx.x;
  const int D = a.D, n4 = D / 4;
  const int nz = a.B * a.m;
  float4 v[kVec];
  float ss = 0.f;
  if (row < nz) {
    const int b = row / a.m, j = row % a.m;
    const T* h = reinterpret_cast<const T*>(a.hidden) + ((size_t)b * a.m + j) * D;
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      if (i < n4) {
        v[k] = f4add(load4(h + 4 * i), load4(a.e_depth + (size_t)j * D + 4 * i));
        ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
      }
    }
    ss = block_sum(ss, red);
    const float inv = rsqrtf(ss / D + a.eps);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      if (i < n4) {
        const float4 g = load4(a.g_stage + 4 * i);
        const float4 zv = make_float4(v[k].x * inv * g.x, v[k].y * inv * g.y, v[k].z * inv * g.z,
                                      v[k].w * inv * g.w);
        store4_planes(a.z, a.nz, (size_t)row * D + 4 * i, zv);
        if (a.tap_z) *reinterpret_cast<float4*>(a.tap_z + (size_t)row * D + 4 * i) = zv;
      }
    }
  } else {
    const int lr = row - nz;
    const int b = lr / (a.G + a.K), i0 = lr % (a.G + a.K);  // rows 0..G-1: the group, then placeholders
    int tok = 0;
    if (i0 < a.G) {
      tok = a.anchor[b * a.G + i0];
      if (tok < 0 || tok >= a.V) {
        if (threadIdx.x == 0) flag_status(a.status, kDevBounds);
        tok = 0;
      }
    }
    const T* E = reinterpret_cast<const T*>(a.E);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      if (i < n4) {
        v[k] = (i0 < a.G) ? load4(E + (a.E_tiled ? tiled_index(tok, 4 * i, D) : (size_t)tok * D + 4 * i))
                         : load4(a.e_ph + 4 * i);
        *reinterpret_cast<float4*>(a.x + (size_t)lr * D + 4 * i) = v[k];
        ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
      }
    }
    ss = block_sum(ss, red);
    const float inv = rsqrtf(ss / D + a.eps);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      if (i < n4) {
        const float4 g = load4(a.g_attn0 + 4 * i);
        store4_planes(a.y, a.ny, (size_t)lr * D + 4 * i,
                      make_float4(v[k].x * inv * g.x, v[k].y * inv * g.y, v[k].z * inv * g.z,
                                  v[k].w * inv * g.w));
      }
    }
  }
}

cudaError_t launch_stage(const StageArgs& a, bool f32, cudaStream_t s) {
  const int rows = a.B * a.m + a.B * (a.G + a.K);
  // few rows: 1024 threads per row; many: 256 threads with four float4 of the
  // row each (D <= 4096; few registers, so that every row runs in one wave:
  // 704 rows at B = 32 took two waves of 512-thread CTAs), else 512
  if (rows <= 2 * device_sms() || a.D / 4 > 4 * 256) {
    const int threads = rows <= 2 * device_sms() ? 1024 : 512;
    if (a.D / 4 > kRowVec * threads) return cudaErrorInvalidValue;
    if (f32) return launch_pdl(stage_kernel<float, kRowVec>, dim3(rows), dim3(threads), 0, s, a);
    return launch_pdl(stage_kernel<bf16, kRowVec>, dim3(rows), dim3(threads), 0, s, a);
  }
  if (f32) return launch_pdl(stage_kernel<float, 4>, dim3(rows), dim3(256), 0, s, a);
  return launch_pdl(stage_kernel<bf16, 4>, dim3(rows), dim3(256), 0, s, a);
}

// ---------------------------------------------------------------- K2b: block attention
// One warp-wide bf16 tensor-core product D[16 x 8] += A[16 x 16] B[16 x 8]
// (fp32 accumulation; lane (g, c) = (lane / 4, lane % 4) holds A rows g, g + 8
// at columns 2c, 2c + 1 (+8), B columns g at rows 2c, 2c + 1 (+8), D rows
// g, g + 8 at columns 2c, 2c + 1).
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// One CTA per (hq query heads of one key/value group, request b): with many
// requests hq = n_q / n_kv, so each head's keys and values are reduced from the
// split-K partials once; with few requests hq shrinks to spread the work over
// more SMs (the keys and values are then reduced by each CTA of the group). Sums the QKV partials of the request's rows (4 columns per
// item), applies RoPE to the local queries / keys (table [K+1][d_h/2]), then
// runs non-causal softmax attention of each query row over all m + K + 1 keys:
// one warp per query row, one lane per key for the scores, warp-shuffle
// max / sum, and 4 output columns per lane. Shared rows are d_h + 4 floats so
// 16-byte accesses by 8 consecutive lanes hit distinct banks.
constexpr int kAttnThreads = 512;

// kDepth split loads in flight per item; kMinCtas CTAs per SM (two when the
// grid exceeds the SMs: fewer registers, shallower loads).
template <int kDepth, int kMinCtas>
__global__ void __launch_bounds__(kAttnThreads, kMinCtas) attention_kernel(AttnArgs a) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float sm[];
  const int G = a.hq, g = (int)(blockIdx.x * G) / (a.n_q / a.n_kv), h0 = blockIdx.x * G, b = blockIdx.y;
  const int K1 = a.K1 ? a.K1 : a.K + 1, dh = a.d_h, half = dh / 2;  // local rows (group + placeholders)
  const int qd = a.n_q * dh, kvd = a.n_kv * dh;
  const int ldl = qd + 2 * kvd;               // local partial row width
  const int ldc = a.ldc ? a.ldc : 2 * kvd;     // context partial row width
  const int Tk = a.m + K1;
  const int LD = dh + 4, LP = 36;
  const int QR = G * K1, QRp = (QR + 15) / 16 * 16, Tkp = (Tk + 15) / 16 * 16;  // padded to tensor-core tiles
  float* qs = sm;              // [QRp][LD]: query row i of head g G + hh at hh * K1 + i
  float* ks = qs + QRp * LD;   // [Tkp][LD]
  float* vs = ks + Tkp * LD;   // [Tkp][LD]
  float* ps = vs + Tkp * LD;   // [QRp][LP] scores, then probabilities
  const size_t sl = (size_t)(a.loc_rows ? a.loc_rows : a.B * K1) * ldl;
  const size_t sc = (size_t)(a.ctx_rows ? a.ctx_rows : a.B * a.m) * ldc;
  auto rnd4 = [&](float4 v) {
    return a.round_bf16 ? make_float4(round_bf16(v.x), round_bf16(v.y), round_bf16(v.z), round_bf16(v.w)) : v;
  };
  const int h4 = half / 4, d4 = dh / 4;
  const int nq = G * K1 * d4, nk = K1 * d4, nv = K1 * d4, nc = a.m * d4;
  // the source (first split plane, plane stride, planes) and the shared-memory
  // destination of item idx: a float4 of a query, local key / value or context
  // key / value row; values are rounded like the keys and queries (after RoPE)
  auto item = [&](int idx, SplitSrc& src, float*& dst, bool& rnd) {
    int row, col;
    bool ctx = false;
    rnd = false;
    if (idx < nq) {  // queries of the group's heads (rotated below)
      const int d = (idx % d4) * 4, r = idx / d4, hh = r / K1;
      row = r % K1, col = (h0 + hh) * dh + d;
      dst = qs + r * LD + d;
    } else if (idx < nq + nk) {  // local keys (rotated below)
      const int t = idx - nq, d = (t % d4) * 4;
      row = t / d4, col = qd + g * dh + d;
      dst = ks + (a.m + row) * LD + d;
    } else if (idx < nq + nk + nv) {  // local values
      const int t = idx - nq - nk, d = (t % d4) * 4;
      row = t / d4, col = qd + kvd + g * dh + d;
      dst = vs + (a.m + row) * LD + d;
      rnd = true;
    } else {  // context keys / values: local position 0, no rotation
      const int t = idx - nq - nk - nv, kv = t / nc, r = t % nc, d = (r % d4) * 4;
      row = r / d4, col = kv * kvd + g * dh + d;
      dst = (kv ? vs : ks) + row * LD + d;
      ctx = true;
      rnd = true;
    }
    if (ctx) {
      const int rr = a.ctx_row0 + b * a.m + row, cc = a.ctx_col0 + col;
      src.p = a.part_ctx + (size_t)rr * ldc + cc;
      src.stride = sc;
      src.n = splits_at(a.sp_ctx, rr, cc);
    } else {
      src.p = a.part_loc + (size_t)(b * K1 + row) * ldl + col;
      src.stride = sl;
      src.n = splits_at(a.sp_loc, b * K1 + row, col);
    }
  };
  // 1) every float4 of the block's rows summed over the split planes, two
  //    items per thread at a time with both items' plane loads in flight
  const int n_items = nq + nk + nv + 2 * nc;
  for (int idx = threadIdx.x; idx < n_items; idx += 2 * blockDim.x) {
    SplitSrc s0, s1;
    float *d0, *d1 = nullptr;
    bool r0, r1 = false;
    item(idx, s0, d0, r0);
    const bool two = idx + (int)blockDim.x < n_items;
    if (two) item(idx + blockDim.x, s1, d1, r1);
    else s1.n = 0;
    float4 v0, v1;
    sum_splits4x2<kDepth>(s0, s1, v0, v1);
    *reinterpret_cast<float4*>(d0) = r0 ? rnd4(v0) : v0;
    if (two) *reinterpret_cast<float4*>(d1) = r1 ? rnd4(v1) : v1;
  }
  __syncthreads();
  // padding rows of the tensor-core tiles hold zeros
  const bool tensor = a.round_bf16 && QR >= 32 && !a.hist_q;
  for (int idx = threadIdx.x; tensor && idx < ((QRp - QR) + 2 * (Tkp - Tk)) * dh; idx += blockDim.x) {
    const int r = idx / dh, d = idx % dh;
    float* row = r < QRp - QR ? qs + (QR + r) * LD
                              : (r < QRp - QR + Tkp - Tk ? ks + (Tk + r - (QRp - QR)) * LD
                                                         : vs + (Tk + r - (QRp - QR) - (Tkp - Tk)) * LD);
    row[d] = 0.f;
  }
  // 2) rotate-half RoPE of the local queries and keys in shared memory
  const int rq = G * K1 * h4, rk = K1 * h4;
  for (int idx = threadIdx.x; idx < rq + rk; idx += blockDim.x) {
    const int t = idx < rq ? idx : idx - rq, j = (t % h4) * 4, r = t / h4;
    const int i = idx < rq ? r % K1 : r;
    float* row = idx < rq ? qs + r * LD : ks + (a.m + r) * LD;
    const float4 x1 = *reinterpret_cast<const float4*>(row + j), x2 = *reinterpret_cast<const float4*>(row + j + half);
    const float4 c = load4(a.rope_cos + i * half + j), sn = load4(a.rope_sin + i * half + j);
    *reinterpret_cast<float4*>(row + j) =
        rnd4(make_float4(x1.x * c.x - x2.x * sn.x, x1.y * c.y - x2.y * sn.y, x1.z * c.z - x2.z * sn.z,
                         x1.w * c.w - x2.w * sn.w));
    *reinterpret_cast<float4*>(row + j + half) =
        rnd4(make_float4(x2.x * c.x + x1.x * sn.x, x2.y * c.y + x1.y * sn.y, x2.z * c.z + x1.z * sn.z,
                         x2.w * c.w + x1.w * sn.w));
  }
  __syncthreads();
  if (a.hist_q) {  // history mode: the rotated, bf16-rounded block goes to the history kernels
    const int hpg = a.n_q / a.n_kv, hh0 = h0 - g * hpg;
    const size_t bg = (size_t)b * a.n_kv + g;
    auto put4 = [](bf16* dst, const float* src) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      __nv_bfloat162 p[2] = {__floats2bfloat162_rn(v.x, v.y), __floats2bfloat162_rn(v.z, v.w)};
      *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<uint2*>(p);
    };
    for (int idx = threadIdx.x; idx < QR * d4; idx += blockDim.x) {
      const int r = idx / d4, d = (idx % d4) * 4, hh = r / K1, i = r % K1;
      put4(a.hist_q + (bg * hpg * K1 + (size_t)(hh0 + hh) * K1 + i) * dh + d, qs + r * LD + d);
    }
    for (int idx = threadIdx.x; hh0 == 0 && idx < 2 * Tk * d4; idx += blockDim.x) {
      const int kv = idx / (Tk * d4), t = idx % (Tk * d4), j = t / d4, d = (t % d4) * 4;
      put4((kv ? a.hist_v : a.hist_k) + (bg * a.hist_ld + a.hist_off + j) * dh + d, (kv ? vs : ks) + j * LD + d);
    }
    return;
  }

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (tensor) {
    // 3) bf16 operands (every value here is a bf16 rounding) and enough query
    //    rows to fill the tiles (with a few rows the scalar form below is as
    //    fast): S = Q K^T on the
    //    tensor cores, softmax per row, O = P V with P split into two bf16 parts
    //    (P = hi + lo to ~2^-16), fp32 accumulation throughout
    const int gq = lane >> 2, cq = lane & 3;
    const int mtiles = QRp / 16, ntk = (Tk + 7) / 8;
    for (int t = warp; t < mtiles * ntk; t += nw) {
      const int mt = t / ntk, nt = t % ntk;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      const float* qa = qs + (mt * 16 + gq) * LD + 2 * cq;
      const float* kb = ks + (nt * 8 + gq) * LD + 2 * cq;
      for (int k0 = 0; k0 < dh; k0 += 16) {
        const uint32_t A[4] = {pack_bf16x2(qa[k0], qa[k0 + 1]), pack_bf16x2(qa[8 * LD + k0], qa[8 * LD + k0 + 1]),
                               pack_bf16x2(qa[k0 + 8], qa[k0 + 9]),
                               pack_bf16x2(qa[8 * LD + k0 + 8], qa[8 * LD + k0 + 9])};
        mma16816(d, A, pack_bf16x2(kb[k0], kb[k0 + 1]), pack_bf16x2(kb[k0 + 8], kb[k0 + 9]));
      }
      const int r0 = mt * 16 + gq, c0 = nt * 8 + 2 * cq;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = r0 + 8 * (e >> 1), c = c0 + (e & 1);
        ps[r * LP + c] = c < Tk ? d[e] * a.scale : -INFINITY;
      }
    }
    __syncthreads();
    for (int r = warp; r < QR; r += nw) {  // softmax over the Tk <= 32 keys, one warp per row
      const float x = lane < Tk ? ps[r * LP + lane] : -INFINITY;
      const float mx = warp_max(x);
      const float e = lane < Tk ? expf(x - mx) : 0.f;
      const float den = warp_sum(e);
      if (lane < Tkp) ps[r * LP + lane] = e / den;
    }
    __syncthreads();
    const int ntd = dh / 8;
    for (int t = warp; t < mtiles * ntd; t += nw) {
      const int mt = t / ntd, nt = t % ntd;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      const float* pa = ps + (mt * 16 + gq) * LP + 2 * cq;
      const float* vb = vs + 2 * cq * LD + nt * 8 + gq;
      for (int k0 = 0; k0 < Tkp; k0 += 16) {
        const float p[8] = {pa[k0], pa[k0 + 1], pa[8 * LP + k0], pa[8 * LP + k0 + 1],
                            pa[k0 + 8], pa[k0 + 9], pa[8 * LP + k0 + 8], pa[8 * LP + k0 + 9]};
        float lo[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) lo[j] = p[j] - __bfloat162float(__float2bfloat16_rn(p[j]));
        const uint32_t Ahi[4] = {pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]), pack_bf16x2(p[4], p[5]),
                                 pack_bf16x2(p[6], p[7])};
        const uint32_t Alo[4] = {pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]), pack_bf16x2(lo[4], lo[5]),
                                 pack_bf16x2(lo[6], lo[7])};
        const float* v = vb + k0 * LD;
        const uint32_t b0 = pack_bf16x2(v[0], v[LD]), b1 = pack_bf16x2(v[8 * LD], v[9 * LD]);
        mma16816(d, Ahi, b0, b1);
        mma16816(d, Alo, b0, b1);
      }
      const int r0 = mt * 16 + gq, col = nt * 8 + 2 * cq;
#pragma unroll
      for (int hh2 = 0; hh2 < 2; ++hh2) {
        const int r = r0 + 8 * hh2;
        if (r < QR) {
          const int hh = r / K1, i = r % K1;
          const size_t idx = (size_t)(b * K1 + i) * qd + (h0 + hh) * dh + col;
          store_planes(a.o, a.no, idx, d[2 * hh2]);
          store_planes(a.o, a.no, idx + 1, d[2 * hh2 + 1]);
        }
      }
    }
    return;
  }
  for (int r = warp; r < G * K1; r += nw) {
    const int hh = r / K1, i = r % K1;
    const float* q = qs + r * LD;
    float sc_ = -INFINITY;
    if (lane < Tk) {
      const float* k = ks + lane * LD;
      float acc0 = 0.f, acc1 = 0.f;
      for (int d = 0; d < dh; d += 8) {
        const float4 qa = *reinterpret_cast<const float4*>(q + d), ka = *reinterpret_cast<const float4*>(k + d);
        const float4 qb = *reinterpret_cast<const float4*>(q + d + 4), kb = *reinterpret_cast<const float4*>(k + d + 4);
        acc0 = fmaf(qa.x, ka.x, fmaf(qa.y, ka.y, fmaf(qa.z, ka.z, fmaf(qa.w, ka.w, acc0))));
        acc1 = fmaf(qb.x, kb.x, fmaf(qb.y, kb.y, fmaf(qb.z, kb.z, fmaf(qb.w, kb.w, acc1))));
      }
      sc_ = (acc0 + acc1) * a.scale;
    }
    const float mx = warp_max(sc_);
    const float e = (lane < Tk) ? expf(sc_ - mx) : 0.f;
    const float den = warp_sum(e);
    const float pj = e / den;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int jk = 0; jk < Tk; ++jk) {
      const float pk = __shfl_sync(0xffffffffu, pj, jk);  // whole warp
      if (lane < d4) {
        const float4 v = *reinterpret_cast<const float4*>(vs + jk * LD + 4 * lane);
        acc.x = fmaf(pk, v.x, acc.x);
        acc.y = fmaf(pk, v.y, acc.y);
        acc.z = fmaf(pk, v.z, acc.z);
        acc.w = fmaf(pk, v.w, acc.w);
      }
    }
    if (lane < d4) store4_planes(a.o, a.no, (size_t)(b * K1 + i) * qd + (h0 + hh) * dh + 4 * lane, acc);
  }
}

size_t attention_smem(int K1, int m, int d_h, int G) {  // K1 local rows per request
  const int QRp = (G * K1 + 15) / 16 * 16, Tkp = (m + K1 + 15) / 16 * 16;
  return ((size_t)(QRp + 2 * Tkp) * (d_h + 4) + (size_t)QRp * 36) * sizeof(float);
}

int attention_heads_per_cta(int n_q, int n_kv, int B) {
  // aim for at least ~128 CTAs; hq divides the group size n_q / n_kv
  int hq = n_q / n_kv;
  while (hq > 1 && (n_q / hq) * B < 128 && (n_q / n_kv) % (hq / 2) == 0) hq /= 2;
  return hq;
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s) {
  const size_t smem = attention_smem(a.K1 ? a.K1 : a.K + 1, a.m, a.d_h, a.hq);
  const dim3 grid(a.n_q / a.hq, a.B);
  const bool many = (int)(grid.x * grid.y) > device_sms();
  void (*fn)(AttnArgs) = many ? attention_kernel<2, 2> : attention_kernel<4, 1>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attention_kernel<2, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         200 * 1024);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attention_kernel<4, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(fn, grid, dim3(kAttnThreads), smem, s, a);
}

// ---------------------------------------------------------------- residual + RMSNorm
// x[r] += sum_s part[s][r]; then either y = RMSNorm(x) * g (next product's
// input) or, after the last layer, b = RMSNorm(x) * g_final for the
// placeholder rows (the anchor row is dropped). A row is served by a cluster
// of C CTAs (C = 8 when there are few rows, else 1), CTA c taking columns
// [c D / C, (c + 1) D / C) with up to kRowVec float4 per thread and every
// split's load issued before use; the C partial sums of squares are
// exchanged through distributed shared memory and added in rank order, so
// every CTA of the row applies the same scale.
template <int kDepth, int kMinCtas, int kVec>  // split loads in flight; CTAs per SM; float4 per thread
__global__ void __launch_bounds__(kRowThreads, kMinCtas) resnorm_kernel(ResNormArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const uint32_t C = cluster_nctarank(), c = cluster_ctarank();
  const int r = blockIdx.x / (int)C, D = a.D;
  const int n4 = D / 4 / (int)C, i0 = n4 * (int)c;  // this CTA's float4 range [i0, i0 + n4)
  const size_t stride = (size_t)a.rows * D;
  float4 v[kVec];
  float ss = 0.f;
  // every load of the thread first (no store in between that the compiler would
  // have to order them after), then the stores
#pragma unroll
  for (int k = 0; k < kVec; ++k) {
    const int i = i0 + threadIdx.x + k * blockDim.x;
    if (i < i0 + n4) {
      const float4 x = *reinterpret_cast<const float4*>(a.x + (size_t)r * D + 4 * i);
      v[k] = f4add(x, sum_splits4<kDepth>(a.part + (size_t)r * D + 4 * i, stride, splits_at(a.sp, r, 4 * i)));
    }
  }
#pragma unroll
  for (int k = 0; k < kVec; ++k) {
    const int i = i0 + threadIdx.x + k * blockDim.x;
    if (i < i0 + n4) {
      const float4 x = v[k];
      *reinterpret_cast<float4*>(a.x + (size_t)r * D + 4 * i) = x;
      if (a.tap_x) *reinterpret_cast<float4*>(a.tap_x + (size_t)r * D + 4 * i) = x;
      ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
    }
  }
  ss = block_sum(ss, red);  // red[0] = this CTA's partial
  if (C > 1) {
    cluster_sync_all();  // every CTA's partial is in its red[0]
    float t = 0.f;
    for (uint32_t q = 0; q < C; ++q) t += ld_cluster_f32(red, q);
    ss = t;
    cluster_sync_all();  // no CTA leaves while another reads its shared memory
  }
  const float inv = rsqrtf(ss / D + a.eps);
  if (a.final_mode) {
    const int b = r / a.K1, i = r % a.K1;
    if (i < a.G) return;  // the group rows give no output
    const size_t orow = (size_t)(b * (a.K1 - a.G) + (i - a.G)) * D;
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int j = i0 + threadIdx.x + k * blockDim.x;
      if (j < i0 + n4) {
        const float4 g = *reinterpret_cast<const float4*>(a.g + 4 * j);
        const float4 o = make_float4(v[k].x * inv * g.x, v[k].y * inv * g.y, v[k].z * inv * g.z,
                                     v[k].w * inv * g.w);
        *reinterpret_cast<float4*>(a.bout + orow + 4 * j) = o;
        store4_planes(a.bp, 2, orow + 4 * j, o);
        if (a.tap_b) *reinterpret_cast<float4*>(a.tap_b + orow + 4 * j) = o;
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int j = i0 + threadIdx.x + k * blockDim.x;
      if (j < i0 + n4) {
        const float4 g = *reinterpret_cast<const float4*>(a.g + 4 * j);
        store4_planes(a.y, a.ny, (size_t)r * D + 4 * j,
                      make_float4(v[k].x * inv * g.x, v[k].y * inv * g.y, v[k].z * inv * g.z,
                                  v[k].w * inv * g.w));
      }
    }
  }
}

constexpr int kResNormCluster = 8;

cudaError_t launch_resnorm(const ResNormArgs& a, cudaStream_t s) {
  // few rows: a cluster per row, so that more SMs pull the split partials
  const int C = (a.rows * kResNormCluster <= 4 * device_sms() && (a.D / 4) % kResNormCluster == 0) ? kResNormCluster : 1;
  const int n4 = a.D / 4 / C;
  int threads = (n4 + 31) / 32 * 32;
  if (threads > kRowThreads) threads = kRowThreads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.rows * C, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = C;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  // a cluster per row: few CTAs, deep loads (every plane of a few-row product, up
  // to 8, in flight at once); else two CTAs per SM (all rows in one wave)
  if (n4 > threads * (C > 1 ? 1 : kRowVec)) return cudaErrorInvalidValue;
  if (C > 1) return cudaLaunchKernelEx(&cfg, resnorm_kernel<8, 1, 1>, a);
  // one CTA per row: as many float4 per thread as the row needs, so that every
  // split plane's load of them can be in flight at once within the registers
  if (n4 <= 2 * threads) return cudaLaunchKernelEx(&cfg, resnorm_kernel<4, 2, 2>, a);
  return cudaLaunchKernelEx(&cfg, resnorm_kernel<2, 2, kRowVec>, a);
}

// ---------------------------------------------------------------- SwiGLU epilogue
// For products on the pair engine (the one-CTA engine fuses this into its
// epilogue). The gate / up columns are interleaved in blocks of 32: feature f
// has its gate at column 64 (f / 32) + f % 32 and its up 32 columns later.
// a[r, f] = silu(gate) * up, float4 (4 features) per thread.
__global__ void swiglu_kernel(const float* part, Splits sp, int rows, int F, bf16* o0, bf16* o1, int no) {
  pdl_trigger();
  pdl_wait();
  const size_t n4 = (size_t)rows * F / 4, stride = (size_t)rows * 2 * F;
  bf16* outs[2] = {o0, o1};
  for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < n4;
       q += (size_t)gridDim.x * blockDim.x) {
    const size_t idx = 4 * q, r = idx / F, f = idx % F;
    const int cg = (int)(64 * (f / 32) + f % 32);
    const float* p = part + r * 2 * F + cg;
    const float4 g = sum_splits4(p, stride, splits_at(sp, (int)r, cg));
    const float4 u = sum_splits4(p + 32, stride, splits_at(sp, (int)r, cg + 32));
    const float4 v = make_float4(g.x / (1.f + expf(-g.x)) * u.x, g.y / (1.f + expf(-g.y)) * u.y,
                                 g.z / (1.f + expf(-g.z)) * u.z, g.w / (1.f + expf(-g.w)) * u.w);
    store4_planes(outs, no, idx, v);
  }
}

cudaError_t launch_swiglu_interleaved(const float* part, const Splits& sp, int rows, int F, bf16* const* o, int no,
                                      cudaStream_t s) {
  const size_t n4 = (size_t)rows * F / 4;
  int blocks = (int)((n4 + 255) / 256);
  if (blocks > device_sms() * 16) blocks = device_sms() * 16;
  return launch_pdl(swiglu_kernel, dim3(blocks), dim3(256), 0, s, part, sp, rows, F, o[0], o[1], no);
}

// ---------------------------------------------------------------- K3: sequential head chain
// With Q = [Q_b | Q_h] and M = Q_h P (R x R), the head h_i = b_i + P t_i has
// t_1 = tanh(c_1), t_i = tanh(c_i + e_{i-1} + M t_{i-1}) where c_i = Q_b b_i
// and e_i = Q_h b_i come from one product over all rows.
// Persistent cluster kernel, M held in registers: a cluster of kChainCluster
// CTAs serves a group of Bg requests; CTA k owns rows [k*rc, (k+1)*rc) of M
// (rc = R/8) and runs R/32 warps. Warp w owns rows k*rc + 4w + rr (rr < 4);
// its lane L holds M[k*rc + 4w + rr][L + 32j] for j < R/32. A step reads the
// previous state once per warp with conflict-free 32-bit loads (lane L reads
// entries L + 32j), does 4 R/32 FMAs per lane and a reduce-scatter over the
// warp (six shuffles) that leaves row 2*bit4 + bit3 of the lane's index in
// each group of eight lanes; lane L & 7 then sends the new entry to CTA L & 7
// of the cluster (distributed shared memory). One hardware cluster barrier per
// step; the state never leaves the chip.
constexpr int kChainCluster = 8;
constexpr int kChainMaxJ = 16;        // R <= 512
constexpr int kChainMaxClusters = 16;  // clusters per launch (128 CTAs)

__device__ __forceinline__ void st_cluster_f32(uint32_t local_addr, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

template <int NJ>  // R = 32 NJ
__global__ void __launch_bounds__(512, 1) head_chain_kernel(ChainArgs a) {
  pdl_trigger();
  extern __shared__ float sm[];
  constexpr int R = 32 * NJ, rc = R / kChainCluster;
  const int Bg = a.Bg, K = a.K;
  float* tbuf = sm;                    // [2][Bg][R] state, written by every CTA of the cluster
  float* ce = tbuf + 2 * (size_t)Bg * R;  // [Bg][K][rc] (c, e) pairs of this CTA's rows
  const uint32_t rank = cluster_ctarank();
  const int group = blockIdx.x / kChainCluster;
  const int r0 = (int)rank * rc;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  // this lane's entries of M (constant: loaded before waiting for the previous kernel)
  float m[4][NJ];
  {
    const float* src = a.Mt + (size_t)rank * 4 * NJ * R + tid;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr)
#pragma unroll
      for (int j = 0; j < NJ; ++j) m[rr][j] = src[(size_t)(rr * NJ + j) * R];
  }
  pdl_wait();
  // c_i, e_i of this CTA's rows for every (request, step): sum of the split planes
  const size_t stride = (size_t)a.rows * 2 * a.Rp;
  const int n_ce = Bg * K * rc;
  for (int idx = tid; idx < n_ce; idx += blockDim.x) {
    const int r = idx % rc, i = (idx / rc) % K, q = idx / (rc * K);
    const int req = group * Bg + q;
    float c = 0.f, e = 0.f;
    if (req < a.B) {
      const float* p = a.part + (size_t)(req * K + i) * 2 * a.Rp + r0 + r;
      float cc[4] = {0.f, 0.f, 0.f, 0.f}, ee[4] = {0.f, 0.f, 0.f, 0.f};
      for (int sp = 0; sp < a.S; sp += 4) {  // the loads of four planes in flight
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (sp + k < a.S) {
            cc[k] += p[(size_t)(sp + k) * stride];
            ee[k] += p[(size_t)(sp + k) * stride + a.Rp];
          }
        }
      }
      c = (cc[0] + cc[1]) + (cc[2] + cc[3]);
      e = (ee[0] + ee[1]) + (ee[2] + ee[3]);
    }
    ce[2 * (size_t)idx] = c;
    ce[2 * (size_t)idx + 1] = e;
  }
  cluster_sync_all();  // every CTA of the cluster is running before any remote store; ce is visible
  const int nq = min(Bg, a.B - group * Bg);  // live requests of this group
  const bool hi = lane & 16, b3 = lane & 8;
  const int rl = 4 * w + 2 * (int)hi + (int)b3;  // the row this lane's group of eight ends up with
  const int dst = lane & 7;                        // the CTA this lane sends to
  for (int i = 0; i < K; ++i) {
    const float* tprev = tbuf + (size_t)((i - 1) & 1) * Bg * R;
    for (int q0 = 0; q0 < nq; q0 += 4) {  // up to four requests interleaved
      float dot[4] = {0.f, 0.f, 0.f, 0.f};
      if (i > 0) {
        float p[4][4];  // [request][row]
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) p[q][rr] = 0.f;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (q0 + q < nq) {
              const float tv = tprev[(size_t)(q0 + q) * R + lane + 32 * j];
#pragma unroll
              for (int rr = 0; rr < 4; ++rr) p[q][rr] = fmaf(m[rr][j], tv, p[q][rr]);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q0 + q >= nq) break;  // uniform across the warp
          // reduce-scatter: halves of the warp keep rows {0,1} / {2,3}, then quarters one row
          float k0 = hi ? p[q][2] : p[q][0], k1 = hi ? p[q][3] : p[q][1];
          const float s0 = hi ? p[q][0] : p[q][2], s1 = hi ? p[q][1] : p[q][3];
          k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
          k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
          float d = b3 ? k1 : k0;
          d += __shfl_xor_sync(0xffffffffu, b3 ? k0 : k1, 8);
          d += __shfl_xor_sync(0xffffffffu, d, 4);
          d += __shfl_xor_sync(0xffffffffu, d, 2);
          d += __shfl_xor_sync(0xffffffffu, d, 1);
          dot[q] = d;
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (q0 + q >= nq) break;
        const float* cq = ce + 2 * ((size_t)((q0 + q) * K + i) * rc + rl);
        float acc = cq[0];
        if (i > 0) acc += cq[1 - 2 * rc] + dot[q];  // e_{i-1} of the same row
        const float t = tanhf(acc);
        const int row = (group * Bg + q0 + q) * K + i;
        if (dst == 0) a.t[(size_t)row * R + r0 + rl] = t;
        if (dst == 1) store_planes(a.tp, 2, (size_t)row * a.ldt + r0 + rl, t);
        const uint32_t laddr =
            (uint32_t)__cvta_generic_to_shared(tbuf + ((size_t)(i & 1) * Bg + q0 + q) * R + r0 + rl);
        st_cluster_f32(laddr, (uint32_t)dst, t);
      }
    }
    cluster_sync_all();
  }
}

int chain_group_size(int R, int B) {
  (void)R;
  return (B + kChainMaxClusters - 1) / kChainMaxClusters;
}

size_t chain_smem_bytes(int R, int K, int Bg) {
  return (2 * (size_t)Bg * R + 2 * (size_t)Bg * K * (R / kChainCluster)) * sizeof(float);
}

using ChainFn = void (*)(ChainArgs);
static ChainFn chain_fn(int R) {
  switch (R / 32) {
    case 1: return head_chain_kernel<1>;
    case 2: return head_chain_kernel<2>;
    case 3: return head_chain_kernel<3>;
    case 4: return head_chain_kernel<4>;
    case 5: return head_chain_kernel<5>;
    case 6: return head_chain_kernel<6>;
    case 7: return head_chain_kernel<7>;
    case 8: return head_chain_kernel<8>;
    case 9: return head_chain_kernel<9>;
    case 10: return head_chain_kernel<10>;
    case 11: return head_chain_kernel<11>;
    case 12: return head_chain_kernel<12>;
    case 13: return head_chain_kernel<13>;
    case 14: return head_chain_kernel<14>;
    case 15: return head_chain_kernel<15>;
    case 16: return head_chain_kernel<16>;
    default: return nullptr;
  }
}

// Clusters of the chain that are resident at once (at most kChainMaxClusters):
// more would run in a second wave and double the serial time.
static int chain_resident_clusters(ChainFn fn, int R, size_t smem) {
  static int cached[kChainMaxJ + 1] = {};
  const int nj = R / 32;
  if (cached[nj]) return cached[nj];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kChainMaxClusters * kChainCluster, 1, 1);
  cfg.blockDim = dim3(R, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kChainCluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();
    n = kChainMaxClusters;
  }
  cached[nj] = n < kChainMaxClusters ? n : kChainMaxClusters;
  return cached[nj];
}

cudaError_t launch_head_chain(const ChainArgs& a_in, cudaStream_t s) {
  if (a_in.R % 32 || a_in.R < 32 || a_in.R > 32 * kChainMaxJ) return cudaErrorInvalidValue;
  const ChainFn fn = chain_fn(a_in.R);
  static uint32_t attr_done = 0;
  const uint32_t bit = 1u << (a_in.R / 32);
  if (!(attr_done & bit)) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr_done |= bit;
  }
  ChainArgs a = a_in;
  // as many requests per cluster as it takes for every cluster to be resident
  const int fit = chain_resident_clusters(fn, a.R, chain_smem_bytes(a.R, a.K, a.Bg));
  const int bg = (a.B + fit - 1) / fit;
  if (bg > a.Bg && chain_smem_bytes(a.R, a.K, bg) <= 200 * 1024) a.Bg = bg;
  const int groups = (a.B + a.Bg - 1) / a.Bg;
  const size_t smem = chain_smem_bytes(a.R, a.K, a.Bg);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(groups * kChainCluster, 1, 1);
  cfg.blockDim = dim3(a.R, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = kChainCluster;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

// h = b + sum_s part[s] (the P t_i product), kept in fp32 and as two bf16 planes.
__global__ void head_out_kernel(const float* part, int S, int rows, int D, const float* bsrc,
                                float* hs, bf16* h0, bf16* h1, float* tap) {
  pdl_trigger();
  pdl_wait();
  const size_t n = (size_t)rows * D, n4 = n / 4;
  bf16* pl[2] = {h0, h1};
  for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < n4;
       q += (size_t)gridDim.x * blockDim.x) {
    const size_t idx = 4 * q;
    const float4 v = f4add(*reinterpret_cast<const float4*>(bsrc + idx), sum_splits4(part + idx, n, S));
    *reinterpret_cast<float4*>(hs + idx) = v;
    store4_planes(pl, 2, idx, v);
    if (tap) *reinterpret_cast<float4*>(tap + idx) = v;
  }
}

cudaError_t launch_head_out(const float* part, int S, int rows, int D, const float* b, float* hs,
                            bf16* const* hp, float* tap, cudaStream_t s) {
  const size_t n4 = (size_t)rows * D / 4;
  int blocks = (int)((n4 + 255) / 256);
  if (blocks > device_sms() * 8) blocks = device_sms() * 8;
  return launch_pdl(head_out_kernel, dim3(blocks), dim3(256), 0, s, part, S, rows, D, b, hs, hp[0], hp[1], tap);
}

// Split an fp32 tensor into two bf16 planes (used for caller-provided b / hs).
__global__ void split_kernel(const float* src, size_t n, bf16* h0, bf16* h1, float* copy) {
  pdl_trigger();
  pdl_wait();
  bf16* pl[2] = {h0, h1};
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    store_planes(pl, 2, i, src[i]);
    if (copy) copy[i] = src[i];
  }
}

cudaError_t launch_split(const float* src, size_t n, bf16* const* pl, float* copy, cudaStream_t s) {
  int blocks = (int)((n + 255) / 256);
  if (blocks > device_sms() * 8) blocks = device_sms() * 8;
  return launch_pdl(split_kernel, dim3(blocks), dim3(256), 0, s, src, n, pl[0], pl[1], copy);
}

// ---------------------------------------------------------------- K5: greedy verify
// One warp per request: lane i < K compares d_{i+1} with the target's choice at
// input index i; A = position of the first zero in the ballot (K if none).
__global__ void verify_greedy_kernel(VerifyArgs a) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= a.B) return;
  const int K = a.K, KV = a.kv < 0 ? K : a.kv;  // only the first KV candidates are verified
  const int c = (lane < K) ? a.cand[b * K + lane] : 0;
  const int tk = (lane <= KV) ? a.tgt[b * (K + 1) + lane] : 0;
  const unsigned pass = __ballot_sync(0xffffffffu, lane < KV && c == tk);
  const unsigned kmask = (KV >= 32) ? 0xffffffffu : ((1u << KV) - 1u);
  const unsigned fail = ~pass & kmask;
  const int A = fail ? (__ffs(fail) - 1) : KV;
  const int tA = __shfl_sync(0xffffffffu, tk, A);
  if (lane <= K) a.commits[b * (K + 1) + lane] = (lane < A) ? c : (lane == A ? tA : -1);
  if (lane == 0) {
    if (tA < 0 || tA >= a.V) flag_status(a.status, kDevBounds);
    a.accepted[b] = A;
    a.n_commit[b] = A + 1;
    a.next_anchor[b] = tA;
  }
}

cudaError_t launch_verify_greedy(const VerifyArgs& a, cudaStream_t s) {
  const int wpb = 8;
  return launch_pdl(verify_greedy_kernel, dim3((a.B + wpb - 1) / wpb), dim3(wpb * 32), 0, s, a);
}

// ---------------------------------------------------------------- K5: sampling verify
//
// Inverse CDF by exact integer prefix sums: every weight w(v) >= 0 is taken as
// the fixed-point integer floor(w(v) * 2^62) (exact for fp32 weights >= 2^-39),
// so prefix sums are exact and independent of the summation order. The row is
// cut into segments of 128 ids; segment sums and their prefix live in shared
// memory (each CTA of a cluster holding a contiguous range of segments); a
// threshold tau = floor(S * u) is located by a binary search over the segment
// prefix, then one warp scans the 128 ids of that segment. Result: the
// smallest v with prefix(v) > tau, i.e. the inverse CDF at u.

constexpr int kSeg = 128;
constexpr int kMaxSegs = 2048;  // V <= 262144

__device__ __forceinline__ unsigned long long fix62(float w) {
  return w > 0.f ? __float2ull_rz(w * 4611686018427387904.0f) : 0ull;  // 2^62
}
__device__ __forceinline__ unsigned long long fix62d(double w) {
  return w > 0.0 ? __double2ull_rz(w * 4611686018427387904.0) : 0ull;
}

// tau = floor(S * (2y + 1) / 2^24) for the uniform u = (y + 1/2) / 2^23.
__device__ __forceinline__ unsigned long long scaled_threshold(unsigned long long S, uint32_t x) {
  const unsigned long long m = 2ull * (x >> 9) + 1ull;
  const unsigned long long lo = S * m, hi = __umul64hi(S, m);
  return (hi << 40) | (lo >> 24);
}

// Loader of 4 consecutive fixed-point weights starting at v (v % 4 == 0).
struct RowF32 {
  static constexpr int kInFlight = 4;
  const float* row;
  int V;
  struct Raw {
    float4 f;
  };
  __device__ __forceinline__ Raw load(int v) const {
    Raw r;
    if (v + 3 < V) {
      r.f = *reinterpret_cast<const float4*>(row + v);
    } else {
      r.f.x = v < V ? row[v] : 0.f;
      r.f.y = v + 1 < V ? row[v + 1] : 0.f;
      r.f.z = v + 2 < V ? row[v + 2] : 0.f;
      r.f.w = v + 3 < V ? row[v + 3] : 0.f;
    }
    return r;
  }
  __device__ __forceinline__ void fix(int v, const Raw& r, unsigned long long (&w)[4]) const {
    w[0] = v < V ? fix62(r.f.x) : 0ull;
    w[1] = v + 1 < V ? fix62(r.f.y) : 0ull;
    w[2] = v + 2 < V ? fix62(r.f.z) : 0ull;
    w[3] = v + 3 < V ? fix62(r.f.w) : 0ull;
  }
  __device__ __forceinline__ void get4(int v, unsigned long long (&w)[4]) const {
    if (v + 3 < V) {
      const float4 f = *reinterpret_cast<const float4*>(row + v);
      w[0] = fix62(f.x); w[1] = fix62(f.y); w[2] = fix62(f.z); w[3] = fix62(f.w);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = (v + j < V) ? fix62(row[v + j]) : 0ull;
    }
  }
};
struct RowFix {
  static constexpr int kInFlight = 2;
  const unsigned long long* row;
  int V;
  struct Raw {
    unsigned long long w[4];
  };
  __device__ __forceinline__ Raw load(int v) const {
    Raw r;
#pragma unroll
    for (int j = 0; j < 4; ++j) r.w[j] = (v + j < V) ? row[v + j] : 0ull;
    return r;
  }
  __device__ __forceinline__ void fix(int, const Raw& r, unsigned long long (&w)[4]) const {
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = r.w[j];
  }
  __device__ __forceinline__ void get4(int v, unsigned long long (&w)[4]) const {
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = (v + j < V) ? row[v + j] : 0ull;
  }
};

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float row_dot(const VerifyArgs& a, int v, const float* h) {
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

// The part of E[v] . h over columns [lo, hi) (lo % 4 == 0): one warp, 4
// columns per lane per 128, up to 4 raw loads per lane in flight (few
// registers: the verification kernel runs two CTAs per SM).
__device__ __forceinline__ float row_dot_part(const VerifyArgs& a, int v, const float* h, int lo, int hi) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  constexpr int kU = 4;
  for (int d0 = lo + lane * 4; d0 < hi; d0 += 128 * kU) {
    uint2 eb[kU];
    float4 ef[kU], hv[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int d = d0 + 128 * u;
      if (d < hi) {
        hv[u] = *reinterpret_cast<const float4*>(h + d);
        if (a.Ef) ef[u] = *reinterpret_cast<const float4*>(a.Ef + (size_t)v * a.D + d);
        else eb[u] = *reinterpret_cast<const uint2*>(a.Eb + tiled_index(v, d, a.D));
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (d0 + 128 * u < hi) {
        float4 e;
        if (a.Ef) {
          e = ef[u];
        } else {
          const __nv_bfloat162 e01 = *reinterpret_cast<const __nv_bfloat162*>(&eb[u].x);
          const __nv_bfloat162 e23 = *reinterpret_cast<const __nv_bfloat162*>(&eb[u].y);
          e = make_float4(__low2float(e01), __high2float(e01), __low2float(e23), __high2float(e23));
        }
        acc = fmaf(e.x, hv[u].x, fmaf(e.y, hv[u].y, fmaf(e.z, hv[u].z, fmaf(e.w, hv[u].w, acc))));
      }
    }
  }
  return warp_sum(acc);
}

// ---- cluster form: the row of one request is cut among kVerifyCluster CTAs

constexpr int kVerifyCluster = 8;
constexpr int kVerifyCThreads = 512;
constexpr int kSegsPerCta = kMaxSegs / kVerifyCluster;

__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_f64(uint32_t addr, double v) {
  asm volatile("st.shared::cluster.f64 [%0], %1;" ::"r"(addr), "d"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Inverse CDF of a row over the cluster: CTA `rank` owns segments
// [rank nseg / C, (rank + 1) nseg / C); the CTAs exchange their totals, so each
// knows S and the prefix before its range, and the CTA whose range holds a
// threshold resolves it and writes the id into out[j] of cluster rank 0.
// xs (nthr <= 32 words) must be identical in every CTA. Returns S. Must be
// called by every thread of every CTA of the cluster.
template <typename Row, int kC = kVerifyCluster>  // kC CTAs in the cluster
__device__ unsigned long long cluster_icdf(const Row& row, int V, const uint32_t* xs, int nthr, int* out,
                                           unsigned long long* incl, unsigned long long* tot, uint32_t rank) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int nseg = (V + kSeg - 1) / kSeg;
  const int s0 = (int)rank * nseg / kC, s1 = ((int)rank + 1) * nseg / kC;
  const int ns = s1 - s0;
  // 1) segment sums of this CTA's range: one warp per segment, the raw loads
  //    of several segments in flight before any is converted
  constexpr int kInFlight = Row::kInFlight;
  for (int i0 = warp; i0 < ns; i0 += kInFlight * nw) {
    typename Row::Raw raw[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const int i = i0 + u * nw;
      if (i < ns) raw[u] = row.load((s0 + i) * kSeg + lane * 4);
    }
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const int i = i0 + u * nw;
      if (i < ns) {
        unsigned long long w[4];
        row.fix((s0 + i) * kSeg + lane * 4, raw[u], w);
        const unsigned long long t = warp_sum_u64(w[0] + w[1] + w[2] + w[3]);
        if (lane == 0) incl[i] = t;
      }
    }
  }
  __syncthreads();
  // 2) local inclusive scan; 3) the local total into every CTA's tot[rank]
  if (warp == 0) {
    unsigned long long carry = 0;
    for (int base = 0; base < ns; base += 32) {
      const int i = base + lane;
      unsigned long long v = (i < ns) ? incl[i] : 0ull;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (i < ns) incl[i] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane < kC) st_cluster_u64(cluster_addr(tot + rank, (uint32_t)lane), carry);
  }
  cluster_sync_all();
  unsigned long long S = 0, off = 0;
#pragma unroll
  for (int r = 0; r < kC; ++r) {
    if (r < (int)rank) off += tot[r];
    S += tot[r];
  }
  const unsigned long long lt = tot[rank];
  // 4) the thresholds that fall into this CTA's range
  for (int j = warp; j < nthr; j += nw) {
    const unsigned long long tau = scaled_threshold(S, xs[j]);
    if (S == 0ull) {
      if (rank == 0 && lane == 0) out[j] = V - 1;  // no mass: last id (as a plain inverse CDF)
      continue;
    }
    if (tau < off || tau >= off + lt) continue;
    const unsigned long long tl = tau - off;
    int lo = 0, hi = ns - 1;  // first local segment with incl > tl
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (incl[mid] > tl) hi = mid; else lo = mid + 1;
    }
    const unsigned long long before = lo > 0 ? incl[lo - 1] : 0ull;
    unsigned long long w[4];
    row.get4((s0 + lo) * kSeg + lane * 4, w);
    const unsigned long long mine = w[0] + w[1] + w[2] + w[3];
    unsigned long long pre = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long u = __shfl_up_sync(0xffffffffu, pre, o);
      if (lane >= o) pre += u;
    }
    const unsigned long long start = before + pre - mine;
    const unsigned ball = __ballot_sync(0xffffffffu, start + mine > tl);
    const int L = ball ? __ffs(ball) - 1 : 31;
    if (lane == L) {
      unsigned long long c = start;
      int k = 0;
      for (; k < 3; ++k) {
        c += w[k];
        if (c > tl) break;
      }
      st_cluster_u32(cluster_addr(out + j, 0), (uint32_t)min((s0 + lo) * kSeg + lane * 4 + k, V - 1));
    }
  }
  cluster_sync_all();  // every id is in rank 0's out[]
  return S;
}

// A cluster of kVerifyCluster CTAs per request.
__global__ void __launch_bounds__(kVerifyCThreads, 2) verify_sample_kernel(VerifyArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned long long incl[kSegsPerCta];
  __shared__ unsigned long long tot[kVerifyCluster];
  __shared__ uint32_t xs[kProposals];      // inverse-CDF words of the proposals
  __shared__ double sacc[kProposals];      // acceptance uniforms of the proposals
  __shared__ double qv[kProposals];        // q(v_j) of the proposals (rank 0)
  __shared__ int sv[kProposals];           // proposal ids (rank 0)
  __shared__ int sA, stok;
  __shared__ float qpart[kVerifyCThreads / 32];
  const uint32_t rank = cluster_ctarank();
  const int b = blockIdx.x / kVerifyCluster, K = a.K, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int KV = a.kv < 0 ? K : a.kv;  // only the first KV candidates are verified
  const int nwarps = blockDim.x >> 5;
  const bool lead = rank == 0;
  const double T = a.T;
  const uint32_t pos0 = (uint32_t)a.pos[b];
  const float* prow_base = a.probs + (size_t)b * (K + 1) * a.V;
  if (warp == 0) {  // the accept tests (the same in every CTA of the cluster)
    bool acc = false;
    if (lane < KV) {
      int d = a.cand[b * K + lane];
      if (d < 0 || d >= a.V) {
        if (lead) flag_status(a.status, kDevBounds);
        d = 0;
      }
      const dlite_qstats qs = a.qs[b * K + lane];
      const double q = exp((double)qs.logit / T - (double)qs.lse);
      const uint4 w = philox(0u, pos0 + lane + 1, (uint32_t)b, kTagAccept, a.k0, a.k1);
      const double u = u01d(w.x);
      acc = u * q < (double)prow_base[(size_t)lane * a.V + d];
    }
    const unsigned pass = __ballot_sync(0xffffffffu, acc);
    const unsigned kmask = (KV >= 32) ? 0xffffffffu : ((1u << KV) - 1u);
    const unsigned fail = ~pass & kmask;
    if (lane == 0) sA = fail ? (__ffs(fail) - 1) : KV;
  }
  __syncthreads();
  const int A = sA;
  const float* prow = prow_base + (size_t)A * a.V;
  const RowF32 prow_fix{prow, a.V};
  if (A == KV) {  // every verified draft token accepted: the bonus token from p_KV
    if (threadIdx.x == 0) {
      xs[0] = philox(0u, pos0 + KV + 1, (uint32_t)b, kTagBonus, a.k0, a.k1).x;
      if (lead && a.counters) atomicAdd(a.counters + 3, 1ull);
    }
    __syncthreads();
    cluster_icdf(prow_fix, a.V, xs, 1, sv, incl, tot, rank);
    if (lead && threadIdx.x == 0) stok = sv[0];
  } else {
    const uint32_t posA = pos0 + A + 1;
    if (threadIdx.x < kProposals) {
      const uint4 w = philox((uint32_t)threadIdx.x, posA, (uint32_t)b, kTagResid, a.k0, a.k1);
      xs[threadIdx.x] = w.x;
      sacc[threadIdx.x] = u01d(w.y);
    }
    __syncthreads();
    cluster_icdf(prow_fix, a.V, xs, kProposals, sv, incl, tot, rank);
    // q(v_j) of the proposals, spread over the cluster: CTA r takes proposals
    // r, r + 8, ..., four warps (a quarter of the columns each) per proposal
    const float* h = a.hs + (size_t)(b * K + A) * a.D;
    const double lse_a = (double)a.qs[b * K + A].lse;
    {
      constexpr int kPerCta = kProposals / kVerifyCluster;  // 4
      static_assert(kPerCta * 4 * 32 == kVerifyCThreads, "four warps per proposal");
      const int jj = warp >> 2, qtr = warp & 3;
      const int j = (int)rank + kVerifyCluster * jj;
      const int v = (int)ld_cluster_u32(cluster_addr(sv + j, 0));
      const int qd = ((a.D / 4 + 3) / 4) * 4;  // columns per quarter (a multiple of 4)
      const int lo = min(qtr * qd, a.D), hi = min(lo + qd, a.D);
      const float p = row_dot_part(a, v, h, lo, hi);
      if (lane == 0) qpart[warp] = p;
      __syncthreads();
      if (threadIdx.x < kPerCta) {
        const int jt = (int)rank + kVerifyCluster * (int)threadIdx.x;
        const float* qp = qpart + 4 * threadIdx.x;
        const float l = (qp[0] + qp[1]) + (qp[2] + qp[3]);
        st_cluster_f64(cluster_addr(qv + jt, 0), exp((double)l / T - lse_a));
      }
    }
    cluster_sync_all();
    if (lead && threadIdx.x == 0) {  // proposal-rejection sampling of the residual, in order
      int tok = -1, tried = 0;
      for (int j = 0; j < kProposals; ++j) {
        ++tried;
        const double p = (double)prow[sv[j]];
        if (sacc[j] * p < p - qv[j]) {
          tok = sv[j];
          break;
        }
      }
      if (a.counters) {
        atomicAdd(a.counters + 0, 1ull);
        atomicAdd(a.counters + 1, (unsigned long long)tried);
        if (tok < 0) atomicAdd(a.counters + 2, 1ull);
      }
      for (int r = 0; r < kVerifyCluster; ++r) st_cluster_u32(cluster_addr(&stok, (uint32_t)r), (uint32_t)tok);
    }
    cluster_sync_all();
    if (stok < 0) {
      // exact fallback (rare): inverse CDF over r(v) = max(0, p(v) - q(v)) for all v,
      // each CTA filling the fixed-point residual of its own range of ids
      unsigned long long* r = a.resid + (size_t)b * a.V;
      const int nseg = (a.V + kSeg - 1) / kSeg;
      const int v0 = ((int)rank * nseg / kVerifyCluster) * kSeg;
      const int v1 = min((((int)rank + 1) * nseg / kVerifyCluster) * kSeg, a.V);
      for (int v = v0 + warp; v < v1; v += nwarps) {
        const float l = row_dot(a, v, h);
        if (lane == 0) r[v] = fix62d((double)prow[v] - exp((double)l / T - lse_a));
      }
      __syncthreads();  // this CTA reads back only its own range
      if (threadIdx.x == 0)
        xs[0] = philox((uint32_t)kProposals, posA, (uint32_t)b, kTagResid, a.k0, a.k1).x;
      __syncthreads();
      const RowFix rfix{r, a.V};
      const unsigned long long S = cluster_icdf(rfix, a.V, xs, 1, sv, incl, tot, rank);
      if (S == 0ull) cluster_icdf(prow_fix, a.V, xs, 1, sv, incl, tot, rank);
      if (lead && threadIdx.x == 0) stok = sv[0];
    }
  }
  __syncthreads();
  if (!lead) return;
  const int tok = stok;
  for (int i = threadIdx.x; i <= K; i += blockDim.x)
    a.commits[b * (K + 1) + i] = (i < A) ? a.cand[b * K + i] : (i == A ? tok : -1);
  if (threadIdx.x == 0) {
    if (tok < 0 || tok >= a.V) flag_status(a.status, kDevBounds);
    a.accepted[b] = A;
    a.n_commit[b] = A + 1;
    a.next_anchor[b] = tok;
  }
}

cudaError_t launch_verify_sample(const VerifyArgs& a, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * kVerifyCluster);
  cfg.blockDim = dim3(kVerifyCThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kVerifyCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, verify_sample_kernel, a);
}

constexpr uint32_t kTagMatch = 5;  // Philox tag of the target's own samples (match verification)

// Match verification, step 1: the target's own sample at input index j of
// request b (its choice for position j + 1), for j = 0..kv: inverse CDF over
// p_j with the uniform of Philox(0, pos + j + 1, b, kTagMatch) word 0, one
// cluster of 1-8 CTAs per (request, index) (the same exact fixed-point inverse
// CDF as the sampling verification).
template <int kC>  // CTAs per cluster: fewer when many rows are sampled (one wave)
__global__ void __launch_bounds__(kVerifyCThreads, 2) match_sample_kernel(VerifyArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned long long incl[kMaxSegs / kC];
  __shared__ unsigned long long tot[kC];
  __shared__ uint32_t xs[1];
  __shared__ int sv[1];
  const uint32_t rank = cluster_ctarank();
  const int K = a.K, KV = a.kv < 0 ? K : a.kv;
  const int item = blockIdx.x / kC, b = item / (KV + 1), j = item % (KV + 1);
  const uint32_t pos0 = (uint32_t)a.pos[b];
  if (threadIdx.x == 0) xs[0] = philox(0u, pos0 + j + 1, (uint32_t)b, kTagMatch, a.k0, a.k1).x;
  __syncthreads();
  const RowF32 prow{a.probs + ((size_t)b * (K + 1) + j) * a.V, a.V};
  cluster_icdf<RowF32, kC>(prow, a.V, xs, 1, sv, incl, tot, rank);
  if (rank == 0 && threadIdx.x == 0) a.tsamp[b * (K + 1) + j] = sv[0];
}

template <int kC>
static cudaError_t launch_match_c(const VerifyArgs& a, int items, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(items * kC);
  cfg.blockDim = dim3(kVerifyCThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kC;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, match_sample_kernel<kC>, a);
}

cudaError_t launch_match_sample(const VerifyArgs& a, cudaStream_t s) {
  const int items = a.B * ((a.kv < 0 ? a.K : a.kv) + 1);  // (request, index) rows to sample
  // the largest cluster that keeps every row in one wave (two CTAs per SM)
  const int slots = 2 * device_sms();  // two CTAs per SM: every sampled row in one wave
  if (items * 8 <= slots) return launch_match_c<8>(a, items, s);
  if (items * 4 <= slots) return launch_match_c<4>(a, items, s);
  if (items * 2 <= slots) return launch_match_c<2>(a, items, s);
  return launch_match_c<1>(a, items, s);
}

__global__ void advance_kernel(int B, const int32_t* n_commit, int64_t* pos) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) pos[b] += n_commit[b];
}

cudaError_t launch_advance(int B, const int32_t* n_commit, int64_t* pos, cudaStream_t s) {
  return launch_pdl(advance_kernel, dim3((B + 127) / 128), dim3(128), 0, s, B, n_commit, pos);
}

// The next round's local group: the last G tokens of (group ++ commits[0..n_commit-1]).
__global__ void shift_group_kernel(int B, int G, int K1, const int32_t* commits, const int32_t* n_commit,
                                   int32_t* group) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int n = n_commit[b];
  int32_t* g = group + (size_t)b * G;
  int32_t old[8];
  for (int i = 0; i < G; ++i) old[i] = g[i];
  for (int i = 0; i < G; ++i) {
    const int src = n + i;  // index into (old ++ commits) of length G + n; keep the last G
    g[i] = src < G ? old[src] : commits[(size_t)b * K1 + (src - G)];
  }
}

cudaError_t launch_shift_group(int B, int G, int K1, const int32_t* commits, const int32_t* n_commit,
                               int32_t* group, cudaStream_t s) {
  if (G < 1 || G > 8) return cudaErrorInvalidValue;
  return launch_pdl(shift_group_kernel, dim3((B + 127) / 128), dim3(128), 0, s, B, G, K1, commits, n_commit,
                    group);
}

// ---------------------------------------------------------------- weight preparation

// dst[r][c] = src[r * src_ld + src_off + c] for r < rows, c < cols, converted
// to bf16 planes (two planes: hi / lo) or to fp32.
// dst_ld > 0: row-major planes with row stride dst_ld; dst_ld < 0: tiled planes
// (see tiled_index) with -dst_ld columns.
template <typename T>
__global__ void repack_kernel(const T* src, int rows, int cols, int src_ld, int src_off,
                              bf16* p0, bf16* p1, int np, float* f32, int dst_ld) {
  const size_t n = (size_t)rows * cols;
  bf16* pl[2] = {p0, p1};
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / cols, c = i % cols;
    const float v = to_f32(src[r * src_ld + src_off + c]);
    if (f32) f32[i] = v;
    if (np) {
      const size_t d = dst_ld > 0 ? r * dst_ld + c : tiled_index(r, c, (size_t)(-dst_ld));
      store_planes(pl, np, d, v);
    }
  }
}

cudaError_t launch_repack(const void* src, bool src_f32, int rows, int cols, int src_ld,
                          int src_off, bf16* p0, bf16* p1, int np, float* f32, int dst_ld,
                          cudaStream_t s) {
  const size_t n = (size_t)rows * cols;
  int blocks = (int)((n + 255) / 256);
  if (blocks > device_sms() * 32) blocks = device_sms() * 32;
  if (dst_ld == 0) dst_ld = cols;
  if (src_f32)
    repack_kernel<float><<<blocks, 256, 0, s>>>((const float*)src, rows, cols, src_ld, src_off, p0,
                                                 p1, np, f32, dst_ld);
  else
    repack_kernel<bf16><<<blocks, 256, 0, s>>>((const bf16*)src, rows, cols, src_ld, src_off, p0, p1,
                                                np, f32, dst_ld);
  return cudaGetLastError();
}

// The gate / up weights stacked for the fused SwiGLU epilogue: destination row r
// of [2F, D] is gate row 32 (r / 64) + r % 32 when r % 64 < 32, else up row
// 32 (r / 64) + r % 32; stored in the tiled layout as bf16 planes.
template <typename T>
__global__ void repack_gate_up_kernel(const T* Wg, const T* Wu, int F, int D, bf16* p0, bf16* p1, int np) {
  const size_t n = (size_t)2 * F * D;
  bf16* pl[2] = {p0, p1};
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / D, c = i % D;
    const size_t src_row = 32 * (r / 64) + r % 32;
    const float v = to_f32((r % 64 < 32 ? Wg : Wu)[src_row * D + c]);
    store_planes(pl, np, tiled_index(r, c, (size_t)D), v);
  }
}

cudaError_t launch_repack_gate_up(const void* Wg, const void* Wu, bool src_f32, int F, int D, bf16* p0, bf16* p1,
                                  int np, cudaStream_t s) {
  const size_t n = (size_t)2 * F * D;
  int blocks = (int)((n + 255) / 256);
  if (blocks > device_sms() * 32) blocks = device_sms() * 32;
  if (src_f32)
    repack_gate_up_kernel<float><<<blocks, 256, 0, s>>>((const float*)Wg, (const float*)Wu, F, D, p0, p1, np);
  else
    repack_gate_up_kernel<bf16><<<blocks, 256, 0, s>>>((const bf16*)Wg, (const bf16*)Wu, F, D, p0, p1, np);
  return cudaGetLastError();
}

// M = Q_h P (R x R), float64 accumulate, stored as kChainCluster contiguous
// slices: slice k holds rows [k*R/C, (k+1)*R/C) of M transposed,
// The chain's register image of M: float ((k * 4 R/32 + rr * R/32 + j) * R + 32 w + L)
// holds M[k*R/8 + 4w + rr][L + 32j] for CTA k of the cluster, warp w, lane L.
template <typename T>
__global__ void head_matrix_kernel(const T* Q, const T* P, int D, int R, float* Ms) {
  const int s = blockIdx.x;
  const int rc = R / kChainCluster, nj = R / 32;
  const int L = s & 31, j = s >> 5;
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d)
      acc += (double)to_f32(Q[(size_t)r * 2 * D + D + d]) * (double)to_f32(P[(size_t)d * R + s]);
    const int k = r / rc, rl = r % rc, w = rl >> 2, rr = rl & 3;
    Ms[((size_t)k * 4 * nj + rr * nj + j) * R + 32 * w + L] = (float)acc;
  }
}

cudaError_t launch_head_matrix(const void* Q, const void* P, bool f32, int D, int R, float* Mt,
                               cudaStream_t s) {
  if (f32)
    head_matrix_kernel<float><<<R, 256, 0, s>>>((const float*)Q, (const float*)P, D, R, Mt);
  else
    head_matrix_kernel<bf16><<<R, 256, 0, s>>>((const bf16*)Q, (const bf16*)P, D, R, Mt);
  return cudaGetLastError();
}

}  // namespace dlite
