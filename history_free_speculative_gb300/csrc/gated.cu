// The official gated token-feedback head (a next-step row of the round; the
// round's default head is the low-rank RNN of kernels.cu):
//
//   v_i = E_R(d_{i-1}), d_0 = the anchor;  [g_i, c_i] = W_s [s_{i-1}; v_i] + b_s;
//   f_i = sigmoid(g_i);  s_i = f_i * s_{i-1} + (1 - f_i) * tanh(c_i),  s_0 = 0;
//   r_i = W_h [s_i; u_i] + b_h;  l_i = W_o r_i,
//
// one step at a time because d_i (chosen from l_i) feeds step i + 1. With the
// warm-up (head_warmup), s_0 is one state update from zero on E_R of the token
// before the anchor, with no output ([P1] §"官方顺序头具体算了什么"). The W_h u
// part of all K steps runs once on the tensor-core GEMM engine and the
// vocabulary projection on the LM-head kernel (K = R); each step's state
// update and r are one small kernel each (below).
#include "internal.h"
#include "kernels.h"
#include "tc_device.cuh"

namespace dlite {

namespace {

__device__ __forceinline__ float split_sum(const float* part, size_t stride, int n, size_t idx) {
  float acc = 0.f;
  for (int s = 0; s < n; ++s) acc += part[(size_t)s * stride + idx];  // plane order
  return acc;
}

}  // namespace

// ---------------------------------------------------------------- the step kernels
// With B requests the two step products are B x 2R x 2R (state) and B x R x R
// (r): a few tens of MFMA on weights of 2 MB and 0.5 MB (R = 512, bf16), which
// the vocabulary stream between the steps evicts from L2. Their cost is the
// latency of fetching those weights, so each runs as one small kernel over a
// grid of (FB features) x (4 requests) CTAs whose first act, before waiting
// for the previous kernel, is to request its whole weight slice (FB rows of
// every 64-column tile: one contiguous run each) with bulk copies into shared
// memory; the arithmetic then runs on the CUDA cores from shared memory. The
// state kernel takes the previous token, stages [s_{i-1}; E_R(d_{i-1})], forms
// [g | c] for its FB features and writes s_i; the r kernel forms r_i for its
// FB features. Lane (q, ch) of a warp reads the 16-byte chunk ch of row q of a
// 4-row group (a quarter-warp reads one 128-byte row: no bank conflicts) and
// keeps the partial sums of every (row, request) of its chunks; a reduce-
// scatter over the 8 lanes of a row and a sum over the warps in warp order
// give the products. Weights are read as fp32 (the sum of their bf16 planes).
// The state is double-buffered by step parity: a step reads all of s_{i-1}
// while its CTAs write s_i.
constexpr int kStepRows = 4;   // requests per CTA
constexpr int kStepWarps = 8;  // the warps split the 64-column tiles

namespace {

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&w)[8]) {
  const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    w[2 * e] = __uint_as_float(v[e] << 16);
    w[2 * e + 1] = __uint_as_float(v[e] & 0xffff0000u);
  }
}

// 8 weights of a staged row chunk (np bf16 planes, plane stride in elements) as fp32
template <int NP>
__device__ __forceinline__ void smem_w8(const bf16* w0, size_t plane_stride, float (&w)[8]) {
  bf16x8_to_f32(*reinterpret_cast<const uint4*>(w0), w);
  if (NP == 2) {
    float lo[8];
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(w0 + plane_stride), lo);
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] += lo[e];
  }
}

__device__ __forceinline__ float dot8(const float (&w)[8], const float (&x)[8]) {
  float acc = w[0] * x[0];
#pragma unroll
  for (int e = 1; e < 8; ++e) acc = fmaf(w[e], x[e], acc);
  return acc;
}

// Sum v over the 8 lanes that share lane >> 3, leaving each lane NV / 8 of the
// sums: lane with chunk index ch keeps indices base + k, k < NV / 8, where
// base = (ch >> 2 & 1) NV / 2 + (ch >> 1 & 1) NV / 4 + (ch & 1) NV / 8.
template <int NV>
__device__ __forceinline__ void reduce_scatter8(float (&v)[NV], int ch) {
#pragma unroll
  for (int st = 0; st < 3; ++st) {
    const int half = NV >> (st + 1);
    const int bit = (ch >> (2 - st)) & 1;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float keep = bit ? v[half + k] : v[k];
      const float send = bit ? v[k] : v[half + k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4 >> st);
    }
  }
}

// Request rows r0 .. r0 + FB - 1 of every 64-column tile of a tiled [*, cols]
// matrix (np planes) into dst [plane][tile][FB][64]; thread 0 only.
template <int NP, int FB>
__device__ __forceinline__ void request_slice(const bf16* const* W, int r0, int cols, bf16* dst, uint32_t bar,
                                              int n_tiles_before) {
  const int nkt = cols / 64;
  for (int p = 0; p < NP; ++p)
    for (int t = 0; t < nkt; ++t)
      tc::bulk_load(tc::su32(dst + ((size_t)(p * n_tiles_before) + t) * FB * 64),
                    W[p] + tiled_index((size_t)r0, (size_t)t * 64, (size_t)cols), FB * 128, bar);
}

}  // namespace

// r_i = W_hs s_i + (W_hu u_i) + b_h for features j0 .. j0 + FB - 1 of requests
// b0 .. b0 + nb - 1, from the staged states xs [4][R] (fp32) and the staged
// weight slice wsm [NP][R / 64][FB][64]: kept in fp32 (all steps, for
// verification; this step's, for the exact re-scoring) and as the bf16
// activation of the vocabulary projection. Every thread of the CTA calls it.
template <int NP>
__device__ __forceinline__ void r_product(const GatedArgs& a, int i, const float* xs, const bf16* wsm, float* red,
                                          int j0, int b0, int nb) {
  constexpr int FB = 32 / NP;
  constexpr int NV = FB;  // (FB / 4 rows) x 4 requests
  const int R = a.R, K = a.K, nkt = R / 64;
  const size_t plane = (size_t)nkt * FB * 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = lane >> 3, ch = lane & 7;
  float v[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) v[k] = 0.f;
  for (int t = warp; t < nkt; t += kStepWarps) {
    float x[kStepRows][8];
#pragma unroll
    for (int b = 0; b < kStepRows; ++b) {
      const float4 x0 = *reinterpret_cast<const float4*>(xs + b * R + t * 64 + ch * 8);
      const float4 x1 = *reinterpret_cast<const float4*>(xs + b * R + t * 64 + ch * 8 + 4);
      x[b][0] = x0.x, x[b][1] = x0.y, x[b][2] = x0.z, x[b][3] = x0.w;
      x[b][4] = x1.x, x[b][5] = x1.y, x[b][6] = x1.z, x[b][7] = x1.w;
    }
#pragma unroll
    for (int rg = 0; rg < FB / 4; ++rg) {
      float w[8];
      smem_w8<NP>(wsm + (size_t)t * FB * 64 + (rg * 4 + q) * 64 + ch * 8, plane, w);
#pragma unroll
      for (int b = 0; b < kStepRows; ++b) v[rg * 4 + b] += dot8(w, x[b]);
    }
  }
  reduce_scatter8<NV>(v, ch);
#pragma unroll
  for (int k = 0; k < NV / 8; ++k) {
    const int idx = ((ch >> 2) & 1) * (NV / 2) + ((ch >> 1) & 1) * (NV / 4) + (ch & 1) * (NV / 8) + k;
    red[(warp * FB + (idx / 4) * 4 + q) * kStepRows + idx % 4] = v[k];
  }
  __syncthreads();
  if (threadIdx.x < FB * kStepRows) {
    const int l = threadIdx.x / kStepRows, r = threadIdx.x % kStepRows;
    if (r < nb) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kStepWarps; ++w) acc += red[(w * FB + l) * kStepRows + r];
      const int b = b0 + r, j = j0 + l;
      const size_t row = (size_t)b * K + i - 1;
      acc += a.hu[row * R + j] + a.bh[j];
      a.r_all[row * R + j] = acc;
      a.r_step[(size_t)b * R + j] = acc;
      a.rp[(size_t)b * R + j] = __float2bfloat16_rn(acc);
    }
  }
}

// Step i (0: the warm-up on the token before the anchor, no output; 1: the
// anchor; then the previous step's choice, which is also stored into cand / qs):
// [g | c] = W_s [s_{i-1}; E_R(d_{i-1})] + b_s, s_i = f s_{i-1} + (1 - f) tanh(c).
// kR (one bf16 weight plane): the step's r as well, in the same launch. The
// grid's x extent (R / 32 feature blocks) is then one thread-block cluster:
// every CTA sends its slice of s_i to all CTAs of the cluster (distributed
// shared memory), one cluster barrier, and each CTA forms r for its 32
// features from the whole s_i with its W_hs slice, requested at the start
// with the W_s slice. Same arithmetic and order as the separate r kernel.
// Shared memory: [NP][g | c][2R / 64][FB][64] bf16, (kR) [R / 64][FB][64] bf16,
// [4][2R] fp32 inputs, [8][2][FB][4] fp32 warp sums, (kR) [4][R] fp32 s_i and
// [8][FB][4] fp32 warp sums.
template <int NP, bool kR>
__global__ void __launch_bounds__(kStepWarps * 32) gated_state_kernel(GatedArgs a, int i) {
  static_assert(!kR || NP == 1, "the fused step keeps one weight plane");
  constexpr int FB = 32 / NP;  // features per CTA
  constexpr int NV = 2 * FB;   // partial sums per lane: (g | c) x (FB / 4 rows) x 4 requests
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int tok[kStepRows];
  __shared__ int ok_s;
  const int R = a.R, R2 = 2 * R, K = a.K, nkt = R2 / 64;
  const bool with_r = kR && i >= 1;  // the warm-up step has no output
  bf16* wsm = reinterpret_cast<bf16*>(smem);
  const size_t plane = (size_t)2 * nkt * FB * 64;  // elements per staged plane
  bf16* whs = wsm + NP * plane;                     // (kR) the W_hs slice
  const size_t whs_elems = kR ? (size_t)(R / 64) * FB * 64 : 0;
  float* xs = reinterpret_cast<float*>(whs + whs_elems);
  float* red = xs + kStepRows * R2;
  float* s_all = red + kStepWarps * 2 * FB * kStepRows;  // (kR)
  float* red_r = s_all + kStepRows * R;                 // (kR)
  const int j0 = blockIdx.x * FB, b0 = blockIdx.y * kStepRows;
  const int nb = min(kStepRows, a.B - b0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = lane >> 3, ch = lane & 7;
  const uint32_t bar_a = tc::su32(&bar);
  if (threadIdx.x == 0) {  // the weights do not depend on the previous kernel
    tc::mbar_init(bar_a, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tc::mbar_expect_tx(bar_a, (uint32_t)(NP * 2 * nkt * FB * 128 + (with_r ? (R / 64) * FB * 128 : 0)));
    for (int gc = 0; gc < 2; ++gc)  // g rows j0.., c rows R + j0..
      request_slice<NP, FB>(a.Ws, gc * R + j0, R2, wsm + (size_t)gc * nkt * FB * 64, bar_a, 2 * nkt);
    if (with_r) request_slice<1, FB>(a.Whs, j0, R, whs, bar_a, R / 64);
  }
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x < kStepRows) {
    const int b = b0 + threadIdx.x;
    int d = 0;
    if (b < a.B) {
      d = i == 0 ? a.anchor[b * a.G + a.G - 2] : i == 1 ? a.anchor[b * a.G + a.G - 1] : a.cand_tmp[b];
      if (d < 0 || d >= a.V) {
        flag_status(a.status, kDevBounds);
        d = 0;
      }
    }
    tok[threadIdx.x] = d;
  }
  if (blockIdx.x == 0 && threadIdx.x < nb && i >= 1) {  // the step's bookkeeping, once per request
    const int b = b0 + threadIdx.x;
    if (i > 1) {
      a.cand[b * K + i - 2] = a.cand_tmp[b];
      if (a.qs) a.qs[b * K + i - 2] = a.qs_tmp[b];
    }
    if (a.pos) a.pos_i[b] = a.pos[b] + (i - 1);
  }
  __syncthreads();
  // the state starts with the block (at the warm-up step when there is one)
  const bool fresh = i == 0 || (i == 1 && !a.warm);
  const float* s_prev = a.s + (size_t)((i & 1) ^ 1) * a.B * R;
  for (int e = threadIdx.x; e < kStepRows * R2 / 4; e += blockDim.x) {
    const int r = e / (R2 / 4), k = (e % (R2 / 4)) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < nb) {
      if (k >= R)
        v = *reinterpret_cast<const float4*>(a.ER + (size_t)tok[r] * R + k - R);
      else if (!fresh)
        v = *reinterpret_cast<const float4*>(s_prev + (size_t)(b0 + r) * R + k);
    }
    *reinterpret_cast<float4*>(xs + r * R2 + k) = v;
  }
  if (threadIdx.x == 0) ok_s = tc::mbar_wait(bar_a, 0, a.status);
  __syncthreads();
  // after a wait that gave up (status flagged) the CTA lets its copies land and
  // skips the arithmetic; with the fused r it still takes the cluster barrier
  const bool ok = ok_s != 0;
  if (!ok && threadIdx.x == 0) tc::mbar_wait(bar_a, 0, nullptr);
  if (ok) {
    float v[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) v[k] = 0.f;
    for (int t = warp; t < nkt; t += kStepWarps) {
      float x[kStepRows][8];
#pragma unroll
      for (int b = 0; b < kStepRows; ++b) {
        const float4 x0 = *reinterpret_cast<const float4*>(xs + b * R2 + t * 64 + ch * 8);
        const float4 x1 = *reinterpret_cast<const float4*>(xs + b * R2 + t * 64 + ch * 8 + 4);
        x[b][0] = x0.x, x[b][1] = x0.y, x[b][2] = x0.z, x[b][3] = x0.w;
        x[b][4] = x1.x, x[b][5] = x1.y, x[b][6] = x1.z, x[b][7] = x1.w;
      }
#pragma unroll
      for (int gc = 0; gc < 2; ++gc)
#pragma unroll
        for (int rg = 0; rg < FB / 4; ++rg) {
          float w[8];
          smem_w8<NP>(wsm + ((size_t)gc * nkt + t) * FB * 64 + (rg * 4 + q) * 64 + ch * 8, plane, w);
#pragma unroll
          for (int b = 0; b < kStepRows; ++b) v[(gc * (FB / 4) + rg) * 4 + b] += dot8(w, x[b]);
        }
    }
    reduce_scatter8<NV>(v, ch);
#pragma unroll
    for (int k = 0; k < NV / 8; ++k) {
      const int idx = ((ch >> 2) & 1) * (NV / 2) + ((ch >> 1) & 1) * (NV / 4) + (ch & 1) * (NV / 8) + k;
      const int gc = idx / FB, rg = (idx % FB) / 4, b = idx % 4;
      red[((warp * 2 + gc) * FB + rg * 4 + q) * kStepRows + b] = v[k];
    }
  }
  __syncthreads();
  if (ok && threadIdx.x < FB * kStepRows) {
    const int l = threadIdx.x / kStepRows, r = threadIdx.x % kStepRows;
    float s_new = 0.f;  // rows past the batch contribute zeros to the fused r
    if (r < nb) {
      float g = 0.f, c = 0.f;
#pragma unroll
      for (int w = 0; w < kStepWarps; ++w) {
        g += red[((w * 2 + 0) * FB + l) * kStepRows + r];
        c += red[((w * 2 + 1) * FB + l) * kStepRows + r];
      }
      const int j = j0 + l;
      g += a.bs[j];
      c += a.bs[R + j];
      const float f = 1.f / (1.f + expf(-g));
      const float sp = xs[r * R2 + j];  // s_{i-1}[j] (zero for a fresh state)
      s_new = f * sp + (1.f - f) * tanhf(c);
      a.s[(size_t)(i & 1) * a.B * R + (size_t)(b0 + r) * R + j] = s_new;
    }
    if (with_r) {  // this feature of s_i into every CTA of the cluster
      const uint32_t dst = tc::su32(s_all + r * R + j0 + l);
      for (int rank = 0; rank < (int)gridDim.x; ++rank)
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(tc::map_to_rank(dst, (uint32_t)rank)), "f"(s_new)
                     : "memory");
    }
  }
  if (with_r) {
    tc::cluster_sync_all();  // every slice of s_i has arrived (and no CTA writes remotely any more)
    if (ok) r_product<1>(a, i, s_all, whs, red_r, j0, b0, nb);
  }
}

// The separate r kernel (two weight planes, or no cluster of R / 32 CTAs).
template <int NP>
__global__ void __launch_bounds__(kStepWarps * 32) gated_r_kernel(GatedArgs a, int i) {
  constexpr int FB = 32 / NP;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int ok_s;
  const int R = a.R, nkt = R / 64;
  bf16* wsm = reinterpret_cast<bf16*>(smem);
  const size_t plane = (size_t)nkt * FB * 64;
  float* xs = reinterpret_cast<float*>(smem + NP * plane * 2);
  float* red = xs + kStepRows * R;
  const int j0 = blockIdx.x * FB, b0 = blockIdx.y * kStepRows;
  const int nb = min(kStepRows, a.B - b0);
  const uint32_t bar_a = tc::su32(&bar);
  if (threadIdx.x == 0) {
    tc::mbar_init(bar_a, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tc::mbar_expect_tx(bar_a, (uint32_t)(NP * nkt * FB * 128));
    request_slice<NP, FB>(a.Whs, j0, R, wsm, bar_a, nkt);
  }
  pdl_trigger();
  pdl_wait();
  const float* s_i = a.s + (size_t)(i & 1) * a.B * R;
  for (int e = threadIdx.x; e < kStepRows * R / 4; e += blockDim.x) {
    const int r = e / (R / 4), k = (e % (R / 4)) * 4;
    const float4 v = r < nb ? *reinterpret_cast<const float4*>(s_i + (size_t)(b0 + r) * R + k)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(xs + r * R + k) = v;
  }
  if (threadIdx.x == 0) ok_s = tc::mbar_wait(bar_a, 0, a.status);
  __syncthreads();
  if (!ok_s) {
    if (threadIdx.x == 0) tc::mbar_wait(bar_a, 0, nullptr);
    return;
  }
  r_product<NP>(a, i, xs, wsm, red, j0, b0, nb);
}

// out[r][c] = sum of the split planes of a rows x cols product
__global__ void gated_sum_kernel(const float* part, Splits sp, int rows, int cols, float* out) {
  pdl_trigger();
  pdl_wait();
  const size_t n = (size_t)rows * cols, stride = n;
  for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < n; q += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(q / cols), c = (int)(q % cols);
    out[q] = split_sum(part, stride, splits_at(sp, r, c), q);
  }
}

// the last step's choice into cand / qs
__global__ void gated_final_kernel(GatedArgs a) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.B) return;
  a.cand[b * a.K + a.K - 1] = a.cand_tmp[b];
  if (a.qs) a.qs[b * a.K + a.K - 1] = a.qs_tmp[b];
}

static size_t state_smem(int R, int np, bool fused) {
  const int fb = 32 / np;
  size_t b = (size_t)np * 2 * (2 * R / 64) * fb * 128 + (size_t)kStepRows * 2 * R * 4 +
             (size_t)kStepWarps * 2 * fb * kStepRows * 4;
  if (fused) b += (size_t)(R / 64) * fb * 128 + (size_t)kStepRows * R * 4 + (size_t)kStepWarps * fb * kStepRows * 4;
  return b;
}
static size_t r_smem(int R, int np) {
  const int fb = 32 / np;
  return (size_t)np * (R / 64) * fb * 128 + (size_t)kStepRows * R * 4 + (size_t)kStepWarps * fb * kStepRows * 4;
}

static cudaLaunchConfig_t step_config(const GatedArgs& a, bool fused, size_t sm, cudaStream_t s,
                                      cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.R / (32 / a.np), (a.B + kStepRows - 1) / kStepRows);
  cfg.blockDim = dim3(kStepWarps * 32);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = fused ? a.R / 32 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = fused ? 2 : 1;
  return cfg;
}

int gated_step_clusters(const GatedArgs& a) {
  if (a.np != 1 || a.R > 512 || a.R % 64 || a.B < 1) return 0;
  auto fn = gated_state_kernel<1, true>;
  const size_t sm = state_smem(a.R, 1, true);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) != cudaSuccess ||
      (a.R / 32 > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = step_config(a, true, sm, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_gated_state(const GatedArgs& a, int i, bool fused, cudaStream_t s) {
  if (a.R > 512 || a.R % 64 || a.B < 1 || a.np < 1 || a.np > 2 || (fused && a.np != 1)) return cudaErrorInvalidValue;
  const size_t sm = state_smem(a.R, a.np, fused);
  auto fn = fused ? gated_state_kernel<1, true> : a.np == 1 ? gated_state_kernel<1, false> : gated_state_kernel<2, false>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e == cudaSuccess && fused && a.R / 32 > 8)
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = step_config(a, fused, sm, s, attr);
  return cudaLaunchKernelEx(&cfg, fn, a, i);
}
cudaError_t launch_gated_r(const GatedArgs& a, int i, cudaStream_t s) {
  if (a.R > 512 || a.R % 64 || a.B < 1 || a.np < 1 || a.np > 2) return cudaErrorInvalidValue;
  const size_t sm = r_smem(a.R, a.np);
  auto fn = a.np == 1 ? gated_r_kernel<1> : gated_r_kernel<2>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  return launch_pdl(fn, dim3(a.R / (32 / a.np), (a.B + kStepRows - 1) / kStepRows), dim3(kStepWarps * 32), sm, s,
                    a, i);
}
cudaError_t launch_gated_sum(const float* part, const Splits& sp, int rows, int cols, float* out,
                             cudaStream_t s) {
  const size_t n = (size_t)rows * cols;
  int blocks = (int)((n + 255) / 256);
  if (blocks > device_sms() * 8) blocks = device_sms() * 8;
  return launch_pdl(gated_sum_kernel, dim3(blocks), dim3(256), 0, s, part, sp, rows, cols, out);
}
cudaError_t launch_gated_final(const GatedArgs& a, cudaStream_t s) {
  return launch_pdl(gated_final_kernel, dim3((a.B + 127) / 128), dim3(128), 0, s, a);
}

}  // namespace dlite
