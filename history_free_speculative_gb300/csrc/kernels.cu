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
      const float v = (i == 0) ? ld_elem<T>(a.E, (size_t)tok * D + d) : a.e_ph[d];
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
// and e_i = Q_h b_i come from one product over all rows. One CTA per request
// runs the K serial steps with the state t in shared memory.
__global__ void head_chain_kernel(ChainArgs a) {
  extern __shared__ float sm[];
  float* tprev = sm;        // [R]
  float* eprev = sm + a.R;  // [R]
  const int b = blockIdx.x, R = a.R;
  const size_t stride = (size_t)a.rows * 2 * R;
  for (int i = 0; i < a.K; ++i) {
    const int row = b * a.K + i;
    const float* p = a.part + (size_t)row * 2 * R;
    float tv[4], ev[4];
    int cnt = 0;
    for (int r = threadIdx.x; r < R; r += blockDim.x, ++cnt) {
      float c = 0.f, e = 0.f;
      for (int s = 0; s < a.S; ++s) {
        c += p[s * stride + r];
        e += p[s * stride + R + r];
      }
      float acc = c;
      if (i > 0) {
        acc += eprev[r];
        float mt = 0.f;
        for (int k = 0; k < R; ++k) mt = fmaf(a.Mt[(size_t)k * R + r], tprev[k], mt);
        acc += mt;
      }
      tv[cnt] = tanhf(acc);
      ev[cnt] = e;
    }
    __syncthreads();
    cnt = 0;
    for (int r = threadIdx.x; r < R; r += blockDim.x, ++cnt) {
      tprev[r] = tv[cnt];
      eprev[r] = ev[cnt];
      a.t[(size_t)row * R + r] = tv[cnt];
      store_planes(a.tp, 2, (size_t)row * a.ldt + r, tv[cnt]);
    }
    __syncthreads();
  }
}

cudaError_t launch_head_chain(const ChainArgs& a, cudaStream_t s) {
  head_chain_kernel<<<a.B, 256, 2 * a.R * sizeof(float), s>>>(a);
  return cudaGetLastError();
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

// Block-wide inverse CDF over one row for up to 32 thresholds at once:
// out[j] = smallest v with prefix(v) > u[j] * total, prefix sums in float64.
// Each thread owns one contiguous chunk; chunk sums are scanned in float64.
template <typename W>
__device__ void block_inverse_cdf(W weight, int V, const double* u, int nthr, int* out,
                                  double* scan) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int chunk = (V + nt - 1) / nt;
  const int v0 = min(V, tid * chunk), v1 = min(V, v0 + chunk);
  double mine = 0.0;
  int lastpos = -1;
  for (int v = v0; v < v1; ++v) {
    const double w = weight(v);
    mine += w;
    if (w > 0.0) lastpos = v;
  }
  scan[tid] = mine;
  __shared__ int last_any;
  if (tid == 0) last_any = -1;
  if (tid < 32) out[tid] = 0x7fffffff;
  __syncthreads();
  if (lastpos >= 0) atomicMax(&last_any, lastpos);
  // inclusive Hillis-Steele scan of chunk sums (nt <= 1024), fixed order
  for (int off = 1; off < nt; off <<= 1) {
    const double v = (tid >= off) ? scan[tid - off] : 0.0;
    __syncthreads();
    scan[tid] += v;
    __syncthreads();
  }
  const double total = scan[nt - 1];
  const double start = scan[tid] - mine;
  for (int j = 0; j < nthr; ++j) {
    const double tau = u[j] * total;
    if (start <= tau && tau < start + mine) {
      double run = start;
      int hit = lastpos;  // rounding guard: the chunk's last positive id
      for (int v = v0; v < v1; ++v) {
        run += weight(v);
        if (run > tau) {
          hit = v;
          break;
        }
      }
      if (hit >= 0) atomicMin(&out[j], hit);
    }
  }
  __syncthreads();
  if (tid < nthr && out[tid] == 0x7fffffff) out[tid] = last_any < 0 ? 0 : last_any;
  __syncthreads();
}

__device__ __forceinline__ float row_dot(const VerifyArgs& a, int v, const float* h) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  if (a.Ef) {
    const float* e = a.Ef + (size_t)v * a.D;
    for (int d = lane; d < a.D; d += 32) acc = fmaf(e[d], h[d], acc);
  } else {
    const bf16* e = a.Eb + (size_t)v * a.D;
    for (int d = lane; d < a.D; d += 32) acc = fmaf(__bfloat162float(e[d]), h[d], acc);
  }
  return warp_sum(acc);
}

// One CTA per request.
__global__ void verify_sample_kernel(VerifyArgs a) {
  extern __shared__ double dsm[];  // [blockDim.x] scan scratch
  __shared__ int sA, stok;
  __shared__ double su[kProposals];  // inverse-CDF uniforms (proposal draws)
  __shared__ double sacc[kProposals];  // acceptance uniforms of the proposals
  __shared__ double qv[kProposals];  // q(v_j) of the proposals
  __shared__ int sv[32];
  __shared__ double rs;
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
  if (A == K) {
    if (threadIdx.x == 0) {
      const uint4 w = philox(0u, pos0 + K + 1, (uint32_t)b, kTagBonus, a.k0, a.k1);
      su[0] = u01d(w.x);
    }
    __syncthreads();
    block_inverse_cdf([&](int v) { return (double)prow[v]; }, a.V, su, 1, sv, dsm);
    if (threadIdx.x == 0) stok = sv[0];
  } else {
    const uint32_t posA = pos0 + A + 1;
    if (threadIdx.x < kProposals) {
      const uint4 w = philox((uint32_t)threadIdx.x, posA, (uint32_t)b, kTagResid, a.k0, a.k1);
      su[threadIdx.x] = u01d(w.x);
      sacc[threadIdx.x] = u01d(w.y);
    }
    __syncthreads();
    block_inverse_cdf([&](int v) { return (double)prow[v]; }, a.V, su, kProposals, sv, dsm);
    const float* h = a.hs + (size_t)(b * K + A) * a.D;
    const double lse_a = (double)a.qs[b * K + A].lse;
    for (int j = warp; j < kProposals; j += nwarps) {  // one warp per proposal
      const float l = row_dot(a, sv[j], h);
      if (lane == 0) qv[j] = exp((double)l / T - lse_a);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int tok = -1;
      for (int j = 0; j < kProposals; ++j) {
        const double p = (double)prow[sv[j]];
        if (sacc[j] * p < p - qv[j]) {
          tok = sv[j];
          break;
        }
      }
      stok = tok;
    }
    __syncthreads();
    if (stok < 0) {
      // exact fallback: inverse CDF over r(v) = max(0, p(v) - q(v)) for all v
      double* r = a.resid + (size_t)b * a.V;
      for (int v = warp; v < a.V; v += nwarps) {
        const float l = row_dot(a, v, h);
        if (lane == 0) {
          const double q = exp((double)l / T - lse_a);
          const double d = (double)prow[v] - q;
          r[v] = d > 0.0 ? d : 0.0;
        }
      }
      __syncthreads();
      double part = 0.0;
      for (int v = threadIdx.x; v < a.V; v += blockDim.x) part += r[v];
      dsm[threadIdx.x] = part;
      __syncthreads();
      if (threadIdx.x == 0) {
        double t = 0.0;
        for (int i = 0; i < (int)blockDim.x; ++i) t += dsm[i];
        rs = t;
        const uint4 w = philox((uint32_t)kProposals, posA, (uint32_t)b, kTagResid, a.k0, a.k1);
        su[0] = u01d(w.x);
      }
      __syncthreads();
      if (rs > 0.0)
        block_inverse_cdf([&](int v) { return r[v]; }, a.V, su, 1, sv, dsm);
      else
        block_inverse_cdf([&](int v) { return (double)prow[v]; }, a.V, su, 1, sv, dsm);
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
  const int threads = 256;
  verify_sample_kernel<<<a.B, threads, threads * sizeof(double), s>>>(a);
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
    if (np) store_planes(pl, np, r * dst_ld + c, v);
  }
}

cudaError_t launch_repack(const void* src, bool src_f32, int rows, int cols, int src_ld,
                          int src_off, bf16* p0, bf16* p1, int np, float* f32, int dst_ld,
                          cudaStream_t s) {
  const size_t n = (size_t)rows * cols;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 152 * 32) blocks = 152 * 32;
  if (dst_ld <= 0) dst_ld = cols;
  if (src_f32)
    repack_kernel<float><<<blocks, 256, 0, s>>>((const float*)src, rows, cols, src_ld, src_off, p0,
                                                 p1, np, f32, dst_ld);
  else
    repack_kernel<bf16><<<blocks, 256, 0, s>>>((const bf16*)src, rows, cols, src_ld, src_off, p0, p1,
                                                np, f32, dst_ld);
  return cudaGetLastError();
}

// Mt[s][r] = sum_d Q[r][D + d] * P[d][s]  (M = Q_h P, stored transposed), float64 accumulate.
template <typename T>
__global__ void head_matrix_kernel(const T* Q, const T* P, int D, int R, float* Mt) {
  const int s = blockIdx.x, r0 = threadIdx.x;
  for (int r = r0; r < R; r += blockDim.x) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d)
      acc += (double)to_f32(Q[(size_t)r * 2 * D + D + d]) * (double)to_f32(P[(size_t)d * R + s]);
    Mt[(size_t)s * R + r] = (float)acc;
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
