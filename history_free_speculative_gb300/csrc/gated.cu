// The official gated token-feedback head (a next-step row of the round; the
// round's default head is the low-rank RNN of kernels.cu):
//
//   v_i = E_R(d_{i-1}), d_0 = the anchor;  [g_i, c_i] = W_s [s_{i-1}; v_i] + b_s;
//   f_i = sigmoid(g_i);  s_i = f_i * s_{i-1} + (1 - f_i) * tanh(c_i),  s_0 = 0;
//   r_i = W_h [s_i; u_i] + b_h;  l_i = W_o r_i,
//
// one step at a time because d_i (chosen from l_i) feeds step i + 1. With the
// warm-up (head_warmup), s_0 is one state update from zero on E_R of the token
// before the anchor, with no output ([P1] §"官方顺序头具体算了什么"). The two
// state products and the W_h u part run on the tensor-core GEMM engine, the
// vocabulary projection on the LM-head kernel (K = R); these kernels do the
// gather of E_R rows, the gating and the bookkeeping between them.
#include "internal.h"
#include "kernels.h"

namespace dlite {

namespace {

__device__ __forceinline__ float split_sum(const float* part, size_t stride, int n, size_t idx) {
  float acc = 0.f;
  for (int s = 0; s < n; ++s) acc += part[(size_t)s * stride + idx];  // plane order
  return acc;
}

__device__ __forceinline__ void planes2(bf16* const* pl, size_t i, float v) {
  bf16 hi, lo;
  split_bf16(v, hi, lo);
  pl[0][i] = hi;
  pl[1][i] = lo;
}

}  // namespace

// Step i prep, one CTA per request: the previous token (the anchor at i = 1,
// else the previous step's choice, which is also stored into cand / qs), the
// step's RNG positions, and the product input [s_{i-1}; E_R[d_{i-1}]] as two
// bf16 planes (fp32 precision through the tensor cores). i = 0 is the warm-up
// step: the token before the anchor on the zero state, no bookkeeping.
__global__ void gated_prep_kernel(GatedArgs a, int i) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, R = a.R, K = a.K;
  int d = i == 0 ? a.anchor[b * a.G + a.G - 2] : i == 1 ? a.anchor[b * a.G + a.G - 1] : a.cand_tmp[b];
  if (d < 0 || d >= a.V) {
    if (threadIdx.x == 0) flag_status(a.status, kDevBounds);
    d = 0;
  }
  if (threadIdx.x == 0 && i >= 1) {
    if (i > 1) {
      a.cand[b * K + i - 2] = a.cand_tmp[b];
      if (a.qs) a.qs[b * K + i - 2] = a.qs_tmp[b];
    }
    if (a.pos) a.pos_i[b] = a.pos[b] + (i - 1);
  }
  // the state starts with the block (at the warm-up step when there is one)
  const bool fresh = i == 0 || (i == 1 && !a.warm);
  for (int j = threadIdx.x; j < R; j += blockDim.x) {
    float s = 0.f;
    if (fresh)
      a.s[(size_t)b * R + j] = 0.f;
    else
      s = a.s[(size_t)b * R + j];
    planes2(a.xp, (size_t)b * 2 * R + j, s);
    planes2(a.xp, (size_t)b * 2 * R + R + j, a.ER[(size_t)d * R + j]);
  }
}

// [g | c] = sum of the split planes + b_s; s_i = f s_{i-1} + (1 - f) tanh(c)
__global__ void gated_gate_kernel(GatedArgs a, const float* part, Splits sp) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, R = a.R;
  const size_t stride = (size_t)a.B * 2 * R;
  for (int j = threadIdx.x; j < R; j += blockDim.x) {
    const size_t ig = (size_t)b * 2 * R + j, ic = ig + R;
    const float g = split_sum(part, stride, splits_at(sp, b, j), ig) + a.bs[j];
    const float c = split_sum(part, stride, splits_at(sp, b, R + j), ic) + a.bs[R + j];
    const float f = 1.f / (1.f + expf(-g));
    const float s = f * a.s[(size_t)b * R + j] + (1.f - f) * tanhf(c);
    a.s[(size_t)b * R + j] = s;
    planes2(a.sp, (size_t)b * R + j, s);
  }
}

// r_i = W_hs s_i (split planes) + (W_hu u_i) + b_h: kept in fp32 (all steps, for
// verification; this step's, for the exact re-scoring) and as the bf16
// activation of the vocabulary projection
__global__ void gated_r_kernel(GatedArgs a, int i, const float* part, Splits sp) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x, R = a.R, K = a.K;
  const size_t stride = (size_t)a.B * R;
  for (int j = threadIdx.x; j < R; j += blockDim.x) {
    const size_t row = (size_t)b * K + i - 1;
    const float r = split_sum(part, stride, splits_at(sp, b, j), (size_t)b * R + j) + a.hu[row * R + j] + a.bh[j];
    a.r_all[row * R + j] = r;
    a.r_step[(size_t)b * R + j] = r;
    a.rp[(size_t)b * R + j] = __float2bfloat16_rn(r);
  }
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

static int gated_threads(int R) { return R >= 512 ? 512 : (R + 31) / 32 * 32; }

cudaError_t launch_gated_prep(const GatedArgs& a, int i, cudaStream_t s) {
  return launch_pdl(gated_prep_kernel, dim3(a.B), dim3(gated_threads(a.R)), 0, s, a, i);
}
cudaError_t launch_gated_gate(const GatedArgs& a, const float* part, const Splits& sp, cudaStream_t s) {
  return launch_pdl(gated_gate_kernel, dim3(a.B), dim3(gated_threads(a.R)), 0, s, a, part, sp);
}
cudaError_t launch_gated_r(const GatedArgs& a, int i, const float* part, const Splits& sp, cudaStream_t s) {
  return launch_pdl(gated_r_kernel, dim3(a.B), dim3(gated_threads(a.R)), 0, s, a, i, part, sp);
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
