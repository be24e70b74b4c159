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

// ---------------------------------------------------------------- K1: staging
// Rows [0, B*m): z_{b,j} = RMSNorm(hidden_{b,j} + e_depth_j) * g_stage.
// Rows [B*m, B*m + B*(K+1)): local rows x_{b,0} = E[anchor_b], x_{b,i} = e_ph,
// and y = RMSNorm(x) * g_attn (layer 0 input of the QKV product).
template <typename T>
__global__ void stage_kernel(StageArgs a) {
  extern __shared__ float sv[];
  __shared__ float red[32];
  const int row = blockIdx.x;
  const int D = a.D;
  const int nz = a.B * a.m;
  if (row < nz) {
    const int b = row / a.m, j = row % a.m;
    const T* h = reinterpret_cast<const T*>(a.hidden) + ((size_t)b * a.m + j) * D;
    float ss = 0.f;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
      const float v = to_f32(h[d]) + a.e_depth[(size_t)j * D + d];
      sv[d] = v;
      ss += v * v;
    }
    ss = block_sum(ss, red);
    const float inv = rsqrtf(ss / D + a.eps);
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
      const float zv = sv[d] * inv * a.g_stage[d];
      store_planes(a.z, a.nz, (size_t)row * D + d, zv);
      if (a.tap_z) a.tap_z[(size_t)row * D + d] = zv;
    }
  } else {
    const int lr = row - nz;
    const int b = lr / (a.K + 1), i = lr % (a.K + 1);
    int tok = 0;
    if (i == 0) {
      tok = a.anchor[b];
      if (tok < 0 || tok >= a.V) {
        if (threadIdx.x == 0) flag_status(a.status, kDevBounds);
        tok = 0;
      }
    }
    float ss = 0.f;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
      const float v = (i == 0) ? ld_elem<T>(a.E, a.E_tiled ? tiled_index(tok, d, D) : (size_t)tok * D + d)
                               : a.e_ph[d];
      sv[d] = v;
      a.x[(size_t)lr * D + d] = v;
      ss += v * v;
    }
    ss = block_sum(ss, red);
    const float inv = rsqrtf(ss / D + a.eps);
    for (int d = threadIdx.x; d < D; d += blockDim.x)
      store_planes(a.y, a.ny, (size_t)lr * D + d, sv[d] * inv * a.g_attn0[d]);
  }
}

cudaError_t launch_stage(const StageArgs& a, bool f32, cudaStream_t s) {
  const int rows = a.B * a.m + a.B * (a.K + 1);
  const size_t smem = (size_t)a.D * sizeof(float);
  if (f32)
    stage_kernel<float><<<rows, 256, smem, s>>>(a);
  else
    stage_kernel<bf16><<<rows, 256, smem, s>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- K2b: block attention
// One CTA per (kv head g, request b). Sums the QKV split-K partials of the
// request's rows, applies RoPE to the local queries / keys (table [K+1][d_h/2]),
// then runs non-causal softmax attention of the G*(K+1) query rows of this kv
// head over all m + K + 1 keys, one lane per key, warp-shuffle max / sum.
__global__ void attention_kernel(AttnArgs a) {
  extern __shared__ float sm[];
  const int g = blockIdx.x, b = blockIdx.y;
  const int K1 = a.K + 1, dh = a.d_h, half = dh / 2, G = a.n_q / a.n_kv;
  const int qd = a.n_q * dh, kvd = a.n_kv * dh;
  const int ldl = qd + 2 * kvd;  // local partial row width
  const int ldc = 2 * kvd;       // context partial row width
  const int Tk = a.m + K1;
  const int LD = dh + 1;
  float* qs = sm;                   // [G*K1][LD]
  float* ks = qs + G * K1 * LD;     // [Tk][LD]
  float* vs = ks + Tk * LD;         // [Tk][LD]
  const size_t sl = (size_t)a.B * K1 * ldl, sc = (size_t)a.B * a.m * ldc;

  auto sum_loc = [&](int row, int col) {
    const float* p = a.part_loc + (size_t)(b * K1 + row) * ldl + col;
    float v = 0.f;
    for (int s = 0; s < a.S_loc; ++s) v += p[s * sl];
    return v;
  };
  auto sum_ctx = [&](int row, int col) {
    const float* p = a.part_ctx + (size_t)(b * a.m + row) * ldc + col;
    float v = 0.f;
    for (int s = 0; s < a.S_ctx; ++s) v += p[s * sc];
    return v;
  };
  auto rnd = [&](float v) { return a.round_bf16 ? round_bf16(v) : v; };

  // queries: (i, hh, j) pairs
  for (int idx = threadIdx.x; idx < K1 * G * half; idx += blockDim.x) {
    const int j = idx % half, hh = (idx / half) % G, i = idx / (half * G);
    const int col = (g * G + hh) * dh;
    const float x1 = sum_loc(i, col + j), x2 = sum_loc(i, col + j + half);
    const float c = a.rope_cos[i * half + j], sn = a.rope_sin[i * half + j];
    float* q = qs + (hh * K1 + i) * LD;
    q[j] = rnd(x1 * c - x2 * sn);
    q[j + half] = rnd(x2 * c + x1 * sn);
  }
  // local keys (rotated) and values
  for (int idx = threadIdx.x; idx < K1 * half; idx += blockDim.x) {
    const int j = idx % half, i = idx / half;
    const int col = qd + g * dh;
    const float x1 = sum_loc(i, col + j), x2 = sum_loc(i, col + j + half);
    const float c = a.rope_cos[i * half + j], sn = a.rope_sin[i * half + j];
    float* k = ks + (a.m + i) * LD;
    k[j] = rnd(x1 * c - x2 * sn);
    k[j + half] = rnd(x2 * c + x1 * sn);
  }
  for (int idx = threadIdx.x; idx < K1 * dh; idx += blockDim.x) {
    const int d = idx % dh, i = idx / dh;
    vs[(a.m + i) * LD + d] = rnd(sum_loc(i, qd + kvd + g * dh + d));
  }
  // context keys / values: local position 0, no rotation
  for (int idx = threadIdx.x; idx < a.m * dh; idx += blockDim.x) {
    const int d = idx % dh, j = idx / dh;
    ks[j * LD + d] = rnd(sum_ctx(j, g * dh + d));
    vs[j * LD + d] = rnd(sum_ctx(j, kvd + g * dh + d));
  }
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int qr = warp; qr < G * K1; qr += nw) {
    const int hh = qr / K1, i = qr % K1;
    const float* q = qs + qr * LD;
    float sc_ = -INFINITY;
    if (lane < Tk) {
      const float* k = ks + lane * LD;
      float acc = 0.f;
      for (int d = 0; d < dh; ++d) acc = fmaf(q[d], k[d], acc);
      sc_ = acc * a.scale;
    }
    const float mx = warp_max(sc_);
    const float e = (lane < Tk) ? expf(sc_ - mx) : 0.f;
    const float den = warp_sum(e);
    const float pj = e / den;
    const size_t orow = (size_t)(b * K1 + i) * qd + (g * G + hh) * dh;
    for (int d = lane; d < dh; d += 32) {
      float acc = 0.f;
      for (int jk = 0; jk < Tk; ++jk) acc = fmaf(__shfl_sync(0xffffffffu, pj, jk), vs[jk * LD + d], acc);
      store_planes(a.o, a.no, orow + d, acc);
    }
  }
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s) {
  const int K1 = a.K + 1, G = a.n_q / a.n_kv, Tk = a.m + K1;
  const size_t smem = (size_t)(G * K1 + 2 * Tk) * (a.d_h + 1) * sizeof(float);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         96 * 1024);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  attention_kernel<<<dim3(a.n_kv, a.B), 256, smem, s>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- residual + RMSNorm
// x[r] += sum_s part[s][r]; then either y = RMSNorm(x) * g (next product's
// input) or, after the last layer, b = RMSNorm(x) * g_final for the
// placeholder rows (the anchor row is dropped).
__global__ void resnorm_kernel(ResNormArgs a) {
  extern __shared__ float sv[];
  __shared__ float red[32];
  const int r = blockIdx.x, D = a.D;
  const size_t stride = (size_t)a.rows * D;
  float ss = 0.f;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float v = a.x[(size_t)r * D + d];
    const float* p = a.part + (size_t)r * D + d;
    float acc = 0.f;
    for (int s = 0; s < a.S; ++s) acc += p[s * stride];
    v += acc;
    a.x[(size_t)r * D + d] = v;
    if (a.tap_x) a.tap_x[(size_t)r * D + d] = v;
    sv[d] = v;
    ss += v * v;
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / D + a.eps);
  if (!a.final_mode) {
    for (int d = threadIdx.x; d < D; d += blockDim.x)
      store_planes(a.y, a.ny, (size_t)r * D + d, sv[d] * inv * a.g[d]);
  } else {
    const int b = r / a.K1, i = r % a.K1;
    if (i == 0) return;
    const size_t orow = (size_t)(b * (a.K1 - 1) + (i - 1)) * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
      const float v = sv[d] * inv * a.g[d];
      a.bout[orow + d] = v;
      store_planes(a.bp, 2, orow + d, v);
      if (a.tap_b) a.tap_b[orow + d] = v;
    }
  }
}

cudaError_t launch_resnorm(const ResNormArgs& a, cudaStream_t s) {
  resnorm_kernel<<<a.rows, 256, (size_t)a.D * sizeof(float), s>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- SwiGLU epilogue
// a[r, f] = silu(sum_s part[s][r][f]) * sum_s part[s][r][F + f].
__global__ void swiglu_kernel(const float* part, int S, int rows, int F, bf16* o0, bf16* o1, int no) {
  const size_t n = (size_t)rows * F, stride = (size_t)rows * 2 * F;
  bf16* outs[2] = {o0, o1};
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (size_t)gridDim.x * blockDim.x) {
    const size_t r = idx / F, f = idx % F;
    const float* p = part + r * 2 * F + f;
    float gs = 0.f, us = 0.f;
    for (int s = 0; s < S; ++s) {
      gs += p[s * stride];
      us += p[s * stride + F];
    }
    const float v = gs / (1.f + expf(-gs)) * us;
    store_planes(outs, no, idx, v);
  }
}

cudaError_t launch_swiglu(const float* part, int S, int rows, int F, bf16* const* o, int no,
                          cudaStream_t s) {
  const size_t n = (size_t)rows * F;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  swiglu_kernel<<<blocks, 256, 0, s>>>(part, S, rows, F, o[0], o[1], no);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- K3: sequential head chain
// With Q = [Q_b | Q_h] and M = Q_h P (R x R), the head h_i = b_i + P t_i has
// t_1 = tanh(c_1), t_i = tanh(c_i + e_{i-1} + M t_{i-1}) where c_i = Q_b b_i
// and e_i = Q_h b_i come from one product over all rows.
// Persistent cluster kernel: a cluster of kChainCluster CTAs serves a group of
// Bg requests; CTA k owns rows [k*R/C, (k+1)*R/C) of M, kept in shared memory
// (transposed, so a warp reads consecutive rows), computes those entries of
// t_i for every request of the group and writes them into the state buffer
// of every CTA of the cluster (distributed shared memory). One hardware
// cluster barrier per step; the state never leaves the chip.
constexpr int kChainCluster = 8;
constexpr int kChainThreads = 256;

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t local_addr, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

__global__ void __launch_bounds__(kChainThreads) head_chain_kernel(ChainArgs a) {
  extern __shared__ float sm[];
  const int R = a.R, rc = R / kChainCluster;
  const int Bg = a.Bg;
  float* Ms = sm;                      // [R][rc]: Ms[s][r] = M[r0 + r][s]
  float* tbuf = Ms + (size_t)R * rc;   // [2][Bg][R]
  const uint32_t rank = cluster_ctarank();
  const int group = blockIdx.x / kChainCluster;
  const int r0 = (int)rank * rc;
  {  // this CTA's contiguous slice of M: R * rc floats, float4 loads
    const float4* src = reinterpret_cast<const float4*>(a.Mt + (size_t)rank * R * rc);
    float4* dst = reinterpret_cast<float4*>(Ms);
    const int n4 = R * rc / 4;
#pragma unroll 8
    for (int i = threadIdx.x; i < n4; i += blockDim.x) dst[i] = src[i];
  }
  const int rl = threadIdx.x % rc, ql = threadIdx.x / rc;  // (row, request) of this thread
  const int req = group * Bg + ql;
  const bool active = threadIdx.x < rc * Bg && req < a.B;
  const size_t stride = (size_t)a.rows * 2 * a.Rp;
  float e_prev = 0.f;
  cluster_sync_all();  // every CTA of the cluster is running before any remote store
  for (int i = 0; i < a.K; ++i) {
    float t = 0.f;
    if (active) {
      const int row = req * a.K + i;
      const float* p = a.part + (size_t)row * 2 * a.Rp + r0 + rl;
      float c = 0.f, e = 0.f;
      for (int sp = 0; sp < a.S; ++sp) {
        c += p[sp * stride];
        e += p[sp * stride + a.Rp];
      }
      float acc = c;
      if (i > 0) {
        const float* tp = tbuf + ((size_t)((i - 1) & 1) * Bg + ql) * R;
        float mt = 0.f;
#pragma unroll 4
        for (int k = 0; k < R; k += 4) {
          const float4 tv = *reinterpret_cast<const float4*>(tp + k);
          mt = fmaf(Ms[(size_t)k * rc + rl], tv.x, mt);
          mt = fmaf(Ms[(size_t)(k + 1) * rc + rl], tv.y, mt);
          mt = fmaf(Ms[(size_t)(k + 2) * rc + rl], tv.z, mt);
          mt = fmaf(Ms[(size_t)(k + 3) * rc + rl], tv.w, mt);
        }
        acc += e_prev + mt;
      }
      t = tanhf(acc);
      e_prev = e;
      a.t[(size_t)row * R + r0 + rl] = t;
      store_planes(a.tp, 2, (size_t)row * a.ldt + r0 + rl, t);
      const uint32_t laddr = (uint32_t)__cvta_generic_to_shared(
          tbuf + ((size_t)(i & 1) * Bg + ql) * R + r0 + rl);
      for (int k = 0; k < kChainCluster; ++k) st_cluster_f32(laddr, (uint32_t)k, t);
    }
    cluster_sync_all();
  }
}

cudaError_t launch_head_chain(const ChainArgs& a, cudaStream_t s) {
  const int rc = a.R / kChainCluster;
  const int groups = (a.B + a.Bg - 1) / a.Bg;
  const size_t smem = ((size_t)a.R * rc + 2 * (size_t)a.Bg * a.R) * sizeof(float);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(head_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         200 * 1024);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(groups * kChainCluster, 1, 1);
  cfg.blockDim = dim3(kChainThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = kChainCluster;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, head_chain_kernel, a);
}

int chain_group_size(int R, int B) {
  const int rc = R / kChainCluster;
  int bg = kChainThreads / rc;
  if (bg < 1) bg = 1;
  if (bg > B) bg = B;
  return bg;
}

size_t chain_smem_bytes(int R, int Bg) {
  return ((size_t)R * (R / kChainCluster) + 2 * (size_t)Bg * R) * sizeof(float);
}

// h = b + sum_s part[s] (the P t_i product), kept in fp32 and as two bf16 planes.
__global__ void head_out_kernel(const float* part, int S, int rows, int D, const float* bsrc,
                                float* hs, bf16* h0, bf16* h1, float* tap) {
  const size_t n = (size_t)rows * D;
  bf16* pl[2] = {h0, h1};
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (size_t)gridDim.x * blockDim.x) {
    float v = bsrc[idx];
    for (int s = 0; s < S; ++s) v += part[s * n + idx];
    hs[idx] = v;
    store_planes(pl, 2, idx, v);
    if (tap) tap[idx] = v;
  }
}

cudaError_t launch_head_out(const float* part, int S, int rows, int D, const float* b, float* hs,
                            bf16* const* hp, float* tap, cudaStream_t s) {
  const size_t n = (size_t)rows * D;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 152 * 8) blocks = 152 * 8;
  head_out_kernel<<<blocks, 256, 0, s>>>(part, S, rows, D, b, hs, hp[0], hp[1], tap);
  return cudaGetLastError();
}

// Split an fp32 tensor into two bf16 planes (used for caller-provided b / hs).
__global__ void split_kernel(const float* src, size_t n, bf16* h0, bf16* h1, float* copy) {
  bf16* pl[2] = {h0, h1};
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    store_planes(pl, 2, i, src[i]);
    if (copy) copy[i] = src[i];
  }
}

cudaError_t launch_split(const float* src, size_t n, bf16* const* pl, float* copy, cudaStream_t s) {
  int blocks = (int)((n + 255) / 256);
  if (blocks > 152 * 8) blocks = 152 * 8;
  split_kernel<<<blocks, 256, 0, s>>>(src, n, pl[0], pl[1], copy);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- K5: greedy verify
// One warp per request: lane i < K compares d_{i+1} with the target's choice at
// input index i; A = position of the first zero in the ballot (K if none).
__global__ void verify_greedy_kernel(VerifyArgs a) {
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= a.B) return;
  const int K = a.K;
  const int c = (lane < K) ? a.cand[b * K + lane] : 0;
  const int tk = (lane <= K) ? a.tgt[b * (K + 1) + lane] : 0;
  const unsigned pass = __ballot_sync(0xffffffffu, lane < K && c == tk);
  const unsigned kmask = (K >= 32) ? 0xffffffffu : ((1u << K) - 1u);
  const unsigned fail = ~pass & kmask;
  const int A = fail ? (__ffs(fail) - 1) : K;
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
  verify_greedy_kernel<<<(a.B + wpb - 1) / wpb, wpb * 32, 0, s>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- K5: sampling verify
//
// Inverse CDF by exact integer prefix sums: every weight w(v) >= 0 is taken as
// the fixed-point integer floor(w(v) * 2^62) (exact for fp32 weights >= 2^-39),
// so prefix sums are exact and independent of the summation order. The row is
// cut into segments of 128 ids; segment sums and their prefix live in shared
// memory; a threshold tau = floor(S * u) is located by a binary search over
// the segment prefix, then one warp scans the 128 ids of that segment.
// Result: the smallest v with prefix(v) > tau, i.e. the inverse CDF at u.

constexpr int kSeg = 128;
constexpr int kVerifyThreads = 1024;
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
  const float* row;
  int V;
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
  const unsigned long long* row;
  int V;
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

// out[j] for thresholds given by 32-bit Philox words xs[j], j < nthr (<= 32).
// incl: shared [kMaxSegs] scratch. Returns the row total through *total.
template <typename Row>
__device__ void block_icdf(const Row& row, int V, const uint32_t* xs, int nthr, int* out,
                           unsigned long long* incl, unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int nseg = (V + kSeg - 1) / kSeg;
  // 1) segment sums: one warp per segment, one float4 per lane
  for (int sg = warp; sg < nseg; sg += nw) {
    unsigned long long w[4];
    row.get4(sg * kSeg + lane * 4, w);
    const unsigned long long t = warp_sum_u64(w[0] + w[1] + w[2] + w[3]);
    if (lane == 0) incl[sg] = t;
  }
  __syncthreads();
  // 2) inclusive scan of the segment sums (warp 0, sequential chunks of 32)
  if (warp == 0) {
    unsigned long long carry = 0;
    for (int base = 0; base < nseg; base += 32) {
      const int i = base + lane;
      unsigned long long v = (i < nseg) ? incl[i] : 0ull;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (i < nseg) incl[i] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) *total = carry;
  }
  __syncthreads();
  const unsigned long long S = *total;
  // 3) one warp per threshold
  for (int j = warp; j < nthr; j += nw) {
    const unsigned long long tau = scaled_threshold(S, xs[j]);
    // first segment with incl > tau (exists when S > 0)
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (incl[mid] > tau) hi = mid; else lo = mid + 1;
    }
    const unsigned long long before = lo > 0 ? incl[lo - 1] : 0ull;
    unsigned long long w[4];
    row.get4(lo * kSeg + lane * 4, w);
    const unsigned long long mine = w[0] + w[1] + w[2] + w[3];
    unsigned long long pre = mine;  // inclusive scan over lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long u = __shfl_up_sync(0xffffffffu, pre, o);
      if (lane >= o) pre += u;
    }
    const unsigned long long start = before + pre - mine;
    const unsigned ball = __ballot_sync(0xffffffffu, start + mine > tau);
    int v = V - 1;
    if (ball) {
      const int L = __ffs(ball) - 1;
      if (lane == L) {
        unsigned long long c = start;
        int k = 0;
        for (; k < 3; ++k) {
          c += w[k];
          if (c > tau) break;
        }
        out[j] = min(lo * kSeg + lane * 4 + k, V - 1);
      }
    } else if (lane == 0) {
      out[j] = v;  // unreachable when S > 0
    }
  }
  __syncthreads();
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

// One CTA (1024 threads) per request.
__global__ void __launch_bounds__(kVerifyThreads) verify_sample_kernel(VerifyArgs a) {
  __shared__ unsigned long long incl[kMaxSegs];
  __shared__ unsigned long long total;
  __shared__ uint32_t xs[kProposals];      // inverse-CDF words of the proposals
  __shared__ double sacc[kProposals];      // acceptance uniforms of the proposals
  __shared__ double qv[kProposals];        // q(v_j) of the proposals
  __shared__ int sv[kProposals];
  __shared__ int sA, stok;
  const int b = blockIdx.x, K = a.K, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const double T = a.T;
  const uint32_t pos0 = (uint32_t)a.pos[b];
  const float* prow_base = a.probs + (size_t)b * (K + 1) * a.V;
  if (warp == 0) {
    bool acc = false;
    if (lane < K) {
      int d = a.cand[b * K + lane];
      if (d < 0 || d >= a.V) {
        flag_status(a.status, kDevBounds);
        d = 0;
      }
      const dlite_qstats qs = a.qs[b * K + lane];
      const double q = exp((double)qs.logit / T - (double)qs.lse);
      const uint4 w = philox(0u, pos0 + lane + 1, (uint32_t)b, kTagAccept, a.k0, a.k1);
      const double u = u01d(w.x);
      acc = u * q < (double)prow_base[(size_t)lane * a.V + d];
    }
    const unsigned pass = __ballot_sync(0xffffffffu, acc);
    const unsigned kmask = (K >= 32) ? 0xffffffffu : ((1u << K) - 1u);
    const unsigned fail = ~pass & kmask;
    if (lane == 0) sA = fail ? (__ffs(fail) - 1) : K;
  }
  __syncthreads();
  const int A = sA;
  const float* prow = prow_base + (size_t)A * a.V;
  const RowF32 prow_fix{prow, a.V};
  if (A == K) {
    if (threadIdx.x == 0) {
      xs[0] = philox(0u, pos0 + K + 1, (uint32_t)b, kTagBonus, a.k0, a.k1).x;
      if (a.counters) atomicAdd(a.counters + 3, 1ull);
    }
    __syncthreads();
    block_icdf(prow_fix, a.V, xs, 1, sv, incl, &total);
    if (threadIdx.x == 0) stok = sv[0];
  } else {
    const uint32_t posA = pos0 + A + 1;
    if (threadIdx.x < kProposals) {
      const uint4 w = philox((uint32_t)threadIdx.x, posA, (uint32_t)b, kTagResid, a.k0, a.k1);
      xs[threadIdx.x] = w.x;
      sacc[threadIdx.x] = u01d(w.y);
    }
    __syncthreads();
    block_icdf(prow_fix, a.V, xs, kProposals, sv, incl, &total);
    const float* h = a.hs + (size_t)(b * K + A) * a.D;
    const double lse_a = (double)a.qs[b * K + A].lse;
    for (int j = warp; j < kProposals; j += nwarps) {  // one warp per proposal
      const float l = row_dot(a, sv[j], h);
      if (lane == 0) qv[j] = exp((double)l / T - lse_a);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int tok = -1, tried = 0;
      for (int j = 0; j < kProposals; ++j) {
        ++tried;
        const double p = (double)prow[sv[j]];
        if (sacc[j] * p < p - qv[j]) {
          tok = sv[j];
          break;
        }
      }
      stok = tok;
      if (a.counters) {
        atomicAdd(a.counters + 0, 1ull);
        atomicAdd(a.counters + 1, (unsigned long long)tried);
        if (tok < 0) atomicAdd(a.counters + 2, 1ull);
      }
    }
    __syncthreads();
    if (stok < 0) {
      // exact fallback: inverse CDF over r(v) = max(0, p(v) - q(v)) for all v (rare)
      unsigned long long* r = a.resid + (size_t)b * a.V;
      for (int v = warp; v < a.V; v += nwarps) {
        const float l = row_dot(a, v, h);
        if (lane == 0) r[v] = fix62d((double)prow[v] - exp((double)l / T - lse_a));
      }
      __syncthreads();
      if (threadIdx.x == 0)
        xs[0] = philox((uint32_t)kProposals, posA, (uint32_t)b, kTagResid, a.k0, a.k1).x;
      __syncthreads();
      const RowFix rfix{r, a.V};
      block_icdf(rfix, a.V, xs, 1, sv, incl, &total);
      if (total == 0ull) block_icdf(prow_fix, a.V, xs, 1, sv, incl, &total);
      if (threadIdx.x == 0) stok = sv[0];
    }
  }
  __syncthreads();
  const int tok = stok;
  for (int i = threadIdx.x; i <= K; i += blockDim.x)
    a.commits[b * (K + 1) + i] = (i < A) ? a.cand[b * K + i] : (i == A ? tok : -1);
  if (threadIdx.x == 0) {
    a.accepted[b] = A;
    a.n_commit[b] = A + 1;
    a.next_anchor[b] = tok;
  }
}

cudaError_t launch_verify_sample(const VerifyArgs& a, cudaStream_t s) {
  verify_sample_kernel<<<a.B, kVerifyThreads, 0, s>>>(a);
  return cudaGetLastError();
}

__global__ void advance_kernel(int B, const int32_t* n_commit, int64_t* pos) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) pos[b] += n_commit[b];
}

cudaError_t launch_advance(int B, const int32_t* n_commit, int64_t* pos, cudaStream_t s) {
  advance_kernel<<<(B + 127) / 128, 128, 0, s>>>(B, n_commit, pos);
  return cudaGetLastError();
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
  if (blocks > 152 * 32) blocks = 152 * 32;
  if (dst_ld == 0) dst_ld = cols;
  if (src_f32)
    repack_kernel<float><<<blocks, 256, 0, s>>>((const float*)src, rows, cols, src_ld, src_off, p0,
                                                 p1, np, f32, dst_ld);
  else
    repack_kernel<bf16><<<blocks, 256, 0, s>>>((const bf16*)src, rows, cols, src_ld, src_off, p0, p1,
                                                np, f32, dst_ld);
  return cudaGetLastError();
}

// M = Q_h P (R x R), float64 accumulate, stored as kChainCluster contiguous
// slices: slice k holds rows [k*R/C, (k+1)*R/C) of M transposed,
// Ms[k][s][r] = M[k*R/C + r][s], the shared-memory image of CTA k of the chain.
template <typename T>
__global__ void head_matrix_kernel(const T* Q, const T* P, int D, int R, float* Ms) {
  const int s = blockIdx.x;
  const int rc = R / kChainCluster;
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d)
      acc += (double)to_f32(Q[(size_t)r * 2 * D + D + d]) * (double)to_f32(P[(size_t)d * R + s]);
    const int k = r / rc, rl = r % rc;
    Ms[((size_t)k * R + s) * rc + rl] = (float)acc;
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
