// Internal declarations shared by the DLite CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dlite.h"
#include "common.cuh"

#include <atomic>
#include <utility>

namespace dlite {

// Streaming multiprocessors of the current device, queried once per device
// (launch shapes and the planners' cost models are sized by it).
inline int device_sms() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Launch with programmatic stream serialization (see pdl_trigger / pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Layout of the fp32 partial products of one GEMM, part[s][rows][outs]: the
// product is the sum of the first n(r, c) planes at (r, c). Uniform split-K
// (N == 0): n = S everywhere. Stream-K (N > 0): tiles of 256 rows x N outputs
// (tile index (r / 256) * slabs + c / N), each tile's kb k blocks in order
// units tile * kb .. tile * kb + kb - 1 of U units shared by G workers, worker
// p owning units [p U / G, (p + 1) U / G); the workers that share a tile write
// planes 0, 1, ... in order.
struct Splits {
  int S = 1;
  int N = 0;
  int slabs = 0, kb = 0, G = 0;
  long long U = 0;
};
__host__ __device__ __forceinline__ long long splits_owner(const Splits& s, long long u) {
  if (s.U * s.G < 0x7fffffffLL)  // the usual sizes: 32-bit arithmetic, the same quotient
    return (long long)(((uint32_t)(u + 1) * (uint32_t)s.G - 1u) / (uint32_t)s.U);
  return ((u + 1) * s.G - 1) / s.U;
}
__host__ __device__ __forceinline__ int splits_at(const Splits& s, int row, int col) {
  if (!s.N) return s.S;
  const long long tile = (long long)(row >> 8) * s.slabs + col / s.N;
  const long long u0 = tile * s.kb;
  return (int)(splits_owner(s, u0 + s.kb - 1) - splits_owner(s, u0) + 1);
}
inline Splits uniform_splits(int S) {
  Splits sp;
  sp.S = S;
  return sp;
}

// LM-head record of a set of vocabulary columns for one row: the 4 best
// (score, id) in descending order (greedy: logit and vocabulary id; sampling:
// the base-2 chunk score log2(sum 2^(logit log2(e) / T)) - log2(-log2 u_k) and
// the 16-id chunk k), from the bf16 product, and the LSE partials of those
// columns in base 2.
constexpr int kTopK = 4;
struct LmRec {
  float sc[kTopK];
  int id[kTopK];
  float m;  // max of logit log2(e) / T over the columns (sampling)
  float s;  // sum of 2^(logit log2(e) / T - m) over the columns (sampling)
};

// Merge of the LM-head records and exact re-scoring of the finalists.
struct LmMergeArgs {
  const LmRec* rec = nullptr;  // [n_tiles][rows]
  int n_tiles = 0, rows = 0, K = 0, D = 0, V = 0;
  float inv_T = 0.f;           // 0 = greedy
  double T = 0.0;              // the temperature (float32 value) for the re-scoring
  uint32_t k0 = 0, k1 = 0;
  const int64_t* pos = nullptr;
  const float* h = nullptr;    // [rows, D] fp32 head states
  const bf16* Eb = nullptr;    // exact LM weights (bf16, tiled layout) ...
  const float* Ef = nullptr;   // ... or fp32
  int32_t* cand = nullptr;
  dlite_qstats* qs = nullptr;
  unsigned long long* counters = nullptr;  // [4] = finalist sets that were close calls
};

cudaError_t launch_lm_merge(const LmMergeArgs& a, cudaStream_t s);

}  // namespace dlite
