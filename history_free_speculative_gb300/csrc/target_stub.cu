// Synthetic target tokens of the acceptance workloads.
//
// This library holds the drafter and the verification rule, not the target
// model. To time whole rounds with a realistic, ragged acceptance, the target's
// greedy choices are drawn on the device from the acceptance model of the
// workloads: at input index j < K the target agrees with the candidate
// d_{j+1} with probability c_j (the per-position conditional acceptance whose
// products give the prefix survival P(A >= k) = prod c_i, [P1]
// §"分布重叠怎样影响平均推进量"), otherwise it picks a uniform id different
// from d_{j+1}; at index K (the bonus position) it picks a uniform id.
#include "kernels.h"

namespace dlite {
namespace {

constexpr uint32_t kTagTarget = 7;

// One CTA: reads the round counter, draws every (request, index) choice, then
// advances the counter. Draws: the words of Philox(0, pos[b] + j + 1, b, 7);
// agreement iff u(w0) < c_j (both exact in fp32); a disagreeing choice is
// (d + 1 + floor(w1 (V - 1) / 2^32)) mod V, the bonus floor(w1 V / 2^32).
__global__ void __launch_bounds__(1024) synthetic_target_kernel(int B, int K, int V, const int32_t* cand,
                                                                const float* accept_c, int n_tables,
                                                                int32_t* round_ctr, uint32_t k0, uint32_t k1,
                                                                const int64_t* pos, int32_t* tgt) {
  pdl_trigger();
  pdl_wait();
  __shared__ int s_round;
  if (threadIdx.x == 0) s_round = round_ctr ? *round_ctr : 0;
  __syncthreads();
  const int tab = (int)((unsigned)s_round % (unsigned)n_tables);
  const float* c = accept_c + (size_t)tab * B * K;
  const int n = B * (K + 1);
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int b = i / (K + 1), j = i - b * (K + 1);
    const uint4 w = philox(0u, (uint32_t)(pos[b] + j + 1), (uint32_t)b, kTagTarget, k0, k1);
    int t;
    if (j == K) {
      t = (int)(((uint64_t)w.y * (uint32_t)V) >> 32);
    } else {
      int d = cand[(size_t)b * K + j];
      d = (d < 0 || d >= V) ? 0 : d;  // candidates come from the draft; keep the output an id
      if (u01f(w.x) < c[(size_t)b * K + j])
        t = d;
      else
        t = (int)(((long long)d + 1 + (long long)(((uint64_t)w.y * (uint32_t)(V - 1)) >> 32)) % V);
    }
    tgt[(size_t)b * (K + 1) + j] = t;
  }
  __syncthreads();
  if (threadIdx.x == 0 && round_ctr) *round_ctr = s_round + 1;
}

}  // namespace
}  // namespace dlite

extern "C" int dlite_synthetic_target(int B, int K, int V, const int32_t* candidates, const float* accept_c,
                                      int n_tables, int32_t* round_counter, uint64_t seed, const int64_t* pos,
                                      int32_t* target_tokens, dlite_stream_t stream) {
  if (!candidates || !accept_c || !pos || !target_tokens) return DLITE_ERR_INVALID_ARG;
  if (B < 1 || K < 1 || K > 31 || V < 2 || n_tables < 1) return DLITE_ERR_INVALID_ARG;
  const int n = B * (K + 1);
  const int threads = n >= 1024 ? 1024 : (n + 31) / 32 * 32;
  const cudaError_t e = dlite::launch_pdl(dlite::synthetic_target_kernel, dim3(1), dim3(threads), 0,
                                          (cudaStream_t)stream, B, K, V, candidates, accept_c, n_tables,
                                          round_counter, (uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32),
                                          pos, target_tokens);
  return e == cudaSuccess ? DLITE_OK : DLITE_ERR_CUDA;
}
