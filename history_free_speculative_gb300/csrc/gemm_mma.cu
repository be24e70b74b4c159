// Weight-streaming GEMM and the LM head with fused argmax / Gumbel-max + LSE,
// on warp-level bf16 tensor-core MMA (m16n8k16, fp32 accumulate).
//
// C[r, o] = sum_k X[r, k] W[o, k]: X = activations (rows = requests x block
// positions), W = nn.Linear weight [out, in]; both operands K-contiguous.
// Split-K writes fp32 partials [split][row][out]; the consumers (fused
// epilogue kernels) reduce the splits in a fixed order, so results are
// deterministic run to run.
#include "internal.h"

namespace dlite {

constexpr int GBM = 64;   // rows per CTA tile
constexpr int GBN = 128;  // outputs per CTA tile
constexpr int GBK = 32;   // k per pipeline stage
constexpr int GST = 3;    // pipeline stages
constexpr int GLD = GBK + 8;  // padded smem row (80 B): conflict-free ldmatrix
constexpr int GTHREADS = 256;
constexpr int kNumSMs = 152;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  const int sz = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(sz));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const bf16* p) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const bf16* p) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(a));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Shared-memory tile set: up to two planes of X and of W per stage.
struct GemmSmem {
  bf16 A[2][GST][GBM][GLD];
  bf16 B[2][GST][GBN][GLD];
};

// CTA main loop over k-tiles [kt0, kt1): acc[mt][nt][4] for the warp's
// 32 x 32 sub-tile (warp wm = warp & 1 -> rows, wn = warp >> 1 -> outputs).
__device__ __forceinline__ void mma_mainloop(GemmSmem& sm, const Planes& X, const Planes& W,
                                             int rows, int outs, int r0, int o0, int kt0,
                                             int kt1, float (&acc)[2][4][4]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp & 1, wn = warp >> 1;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[i][j][k] = 0.f;

  auto load = [&](int stage, int kt) {
    const int kc = kt * GBK;
    {  // X tile: 64 rows x 4 chunks of 8
      const int row = tid >> 2, ch = tid & 3;
      const bool ok = (r0 + row) < rows;
      for (int p = 0; p < X.n; ++p) {
        const bf16* src = ok ? X.p[p] + (size_t)(r0 + row) * X.ld + kc + ch * 8 : X.p[p];
        cp_async16(&sm.A[p][stage][row][ch * 8], src, ok);
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {  // W tile: 128 rows x 4 chunks
      const int idx = tid + i * GTHREADS;
      const int row = idx >> 2, ch = idx & 3;
      const bool ok = (o0 + row) < outs;
      for (int p = 0; p < W.n; ++p) {
        const bf16* src = ok ? W.p[p] + (size_t)(o0 + row) * W.ld + kc + ch * 8 : W.p[p];
        cp_async16(&sm.B[p][stage][row][ch * 8], src, ok);
      }
    }
  };

#pragma unroll
  for (int s = 0; s < GST - 1; ++s) {
    if (kt0 + s < kt1) load(s, kt0 + s);
    cp_async_commit();
  }
  for (int kt = kt0; kt < kt1; ++kt) {
    cp_async_wait<GST - 2>();
    __syncthreads();
    const int nk = kt + GST - 1;
    if (nk < kt1) load((nk - kt0) % GST, nk);
    cp_async_commit();
    const int st = (kt - kt0) % GST;
#pragma unroll
    for (int kk = 0; kk < GBK; kk += 16) {
      // plane products: (x0,w0), (x1,w0), (x0,w1)
      for (int combo = 0; combo < 3; ++combo) {
        const int px = (combo == 1) ? 1 : 0, pw = (combo == 2) ? 1 : 0;
        if (combo == 1 && X.n < 2) continue;
        if (combo == 2 && W.n < 2) continue;
        uint32_t af[2][4], bfr[4][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
          ldsm_x4(af[mt], &sm.A[px][st][wm * 32 + mt * 16 + (lane & 15)][kk + (lane >> 4) * 8]);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
          ldsm_x2(bfr[nt], &sm.B[pw][st][wn * 32 + nt * 8 + (lane & 7)][kk + ((lane >> 3) & 1) * 8]);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) mma_bf16(acc[mt][nt], af[mt], bfr[nt]);
      }
    }
  }
  cp_async_wait<0>();
}

__global__ void __launch_bounds__(GTHREADS) gemm_partial_kernel(GemmArgs a, int kps) {
  extern __shared__ __align__(16) unsigned char smraw[];
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(smraw);
  const int r0 = blockIdx.y * GBM, o0 = blockIdx.x * GBN;
  const int ktot = a.K / GBK;
  const int kt0 = blockIdx.z * kps, kt1 = min(kt0 + kps, ktot);
  float acc[2][4][4];
  mma_mainloop(sm, a.X, a.W, a.rows, a.outs, r0, o0, kt0, kt1, acc);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wm = warp & 1, wn = warp >> 1, g = lane >> 2, t = lane & 3;
  float* out = a.part + (size_t)blockIdx.z * a.rows * a.outs;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = r0 + wm * 32 + mt * 16 + g + hh * 8;
        const int c = o0 + wn * 32 + nt * 8 + 2 * t;
        if (r < a.rows && c < a.outs)
          *reinterpret_cast<float2*>(out + (size_t)r * a.outs + c) =
              make_float2(acc[mt][nt][2 * hh], acc[mt][nt][2 * hh + 1]);
      }
}

int gemm_splits(int rows, int outs, int K) {
  const int tiles = ((outs + GBN - 1) / GBN) * ((rows + GBM - 1) / GBM);
  const int ktot = K / GBK;
  int s = (2 * kNumSMs + tiles - 1) / tiles;
  s = s < 1 ? 1 : s;
  const int smax = ktot / 4 > 0 ? ktot / 4 : 1;
  if (s > smax) s = smax;
  if (s > 16) s = 16;
  return s;
}

size_t gemm_part_elems(int rows, int outs, int K) {
  return (size_t)gemm_splits(rows, outs, K) * rows * outs;
}

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s) {
  const int ktot = a.K / GBK;
  const int kps = (ktot + a.splits - 1) / a.splits;
  dim3 grid((a.outs + GBN - 1) / GBN, (a.rows + GBM - 1) / GBM, a.splits);
  const size_t smem = sizeof(GemmSmem);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_partial_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  gemm_partial_kernel<<<grid, GTHREADS, smem, s>>>(a, kps);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- LM head

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
  s = s * expf(m - mm) + s2 * expf(m2 - mm);
  m = mm;
}

// One CTA: 128 vocabulary ids x 64 rows (row tile blockIdx.y), full D.
// Writes one LmRec per (vocab tile, row).
__global__ void __launch_bounds__(GTHREADS) lm_head_kernel(LmArgs a) {
  extern __shared__ __align__(16) unsigned char smraw[];
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(smraw);
  __shared__ LmRec red[4][GBM];
  const int r0 = blockIdx.y * GBM, o0 = blockIdx.x * GBN;
  float acc[2][4][4];
  mma_mainloop(sm, a.H, a.E, a.rows, a.V, r0, o0, 0, a.D / GBK, acc);

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wm = warp & 1, wn = warp >> 1, g = lane >> 2, t = lane & 3;
  const bool sampling = a.inv_T > 0.f;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int rl = wm * 32 + mt * 16 + g + hh * 8;  // row within tile
      const int r = r0 + rl;
      LmRec best;
      best.best = -INFINITY;
      best.idx = 0x7fffffff;
      best.logit = 0.f;
      best.m = -INFINITY;
      best.s = 0.f;
      uint32_t pos = 0, req = 0;
      if (sampling && r < a.rows) {
        req = (uint32_t)(r / a.K);
        pos = (uint32_t)(a.pos[req] + (r % a.K) + 1);
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int c = o0 + wn * 32 + nt * 8 + 2 * t;  // even vocab id, c and c+1 share a Philox call
        if (c >= a.V) continue;
        const float l0 = acc[mt][nt][2 * hh], l1 = acc[mt][nt][2 * hh + 1];
        if (!sampling) {
          if (better(l0, c, best.best, best.idx)) { best.best = l0; best.idx = c; best.logit = l0; }
          if (c + 1 < a.V && better(l1, c + 1, best.best, best.idx)) {
            best.best = l1; best.idx = c + 1; best.logit = l1;
          }
        } else {
          const uint4 w = philox((uint32_t)c >> 2, pos, req, kTagGumbel, a.k0, a.k1);
          const uint32_t x0 = (c & 2) ? w.z : w.x, x1 = (c & 2) ? w.w : w.y;
          const float s0 = l0 * a.inv_T + gumbel_from_bits(x0);
          if (better(s0, c, best.best, best.idx)) { best.best = s0; best.idx = c; best.logit = l0; }
          float mloc = l0 * a.inv_T, sloc = 1.f;
          if (c + 1 < a.V) {
            const float s1 = l1 * a.inv_T + gumbel_from_bits(x1);
            if (better(s1, c + 1, best.best, best.idx)) { best.best = s1; best.idx = c + 1; best.logit = l1; }
            lse_merge(mloc, sloc, l1 * a.inv_T, 1.f);
          }
          lse_merge(best.m, best.s, mloc, sloc);
        }
      }
      // reduce over the 4 lanes of the quad (same row)
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        LmRec other;
        other.best = __shfl_xor_sync(0xffffffffu, best.best, o);
        other.idx = __shfl_xor_sync(0xffffffffu, best.idx, o);
        other.logit = __shfl_xor_sync(0xffffffffu, best.logit, o);
        other.m = __shfl_xor_sync(0xffffffffu, best.m, o);
        other.s = __shfl_xor_sync(0xffffffffu, best.s, o);
        if (better(other.best, other.idx, best.best, best.idx)) {
          best.best = other.best; best.idx = other.idx; best.logit = other.logit;
        }
        if (sampling) lse_merge(best.m, best.s, other.m, other.s);
      }
      if (t == 0) red[wn][rl] = best;
    }
  __syncthreads();
  if (threadIdx.x < GBM) {
    const int rl = threadIdx.x, r = r0 + rl;
    LmRec best = red[0][rl];
    for (int w = 1; w < 4; ++w) {
      const LmRec o = red[w][rl];
      if (better(o.best, o.idx, best.best, best.idx)) {
        best.best = o.best; best.idx = o.idx; best.logit = o.logit;
      }
      if (sampling) lse_merge(best.m, best.s, o.m, o.s);
    }
    if (r < a.rows) a.rec[(size_t)blockIdx.x * a.rows + r] = best;
  }
}

int lm_tiles(int V) { return (V + GBN - 1) / GBN; }

cudaError_t launch_lm_head(const LmArgs& a, cudaStream_t s) {
  dim3 grid(lm_tiles(a.V), (a.rows + GBM - 1) / GBM, 1);
  const size_t smem = sizeof(GemmSmem);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  lm_head_kernel<<<grid, GTHREADS, smem, s>>>(a);
  return cudaGetLastError();
}

// One warp per row: merge the per-tile records in a fixed order.
__global__ void lm_merge_kernel(const LmRec* rec, int n_tiles, int rows, int K, float inv_T,
                                int32_t* cand, dlite_qstats* qs) {
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const bool sampling = inv_T > 0.f;
  LmRec best;
  best.best = -INFINITY;
  best.idx = 0x7fffffff;
  best.logit = 0.f;
  best.m = -INFINITY;
  best.s = 0.f;
  for (int tI = lane; tI < n_tiles; tI += 32) {
    const LmRec o = rec[(size_t)tI * rows + r];
    if (better(o.best, o.idx, best.best, best.idx)) {
      best.best = o.best; best.idx = o.idx; best.logit = o.logit;
    }
    if (sampling) lse_merge(best.m, best.s, o.m, o.s);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    LmRec other;
    other.best = __shfl_xor_sync(0xffffffffu, best.best, o);
    other.idx = __shfl_xor_sync(0xffffffffu, best.idx, o);
    other.logit = __shfl_xor_sync(0xffffffffu, best.logit, o);
    other.m = __shfl_xor_sync(0xffffffffu, best.m, o);
    other.s = __shfl_xor_sync(0xffffffffu, best.s, o);
    if (better(other.best, other.idx, best.best, best.idx)) {
      best.best = other.best; best.idx = other.idx; best.logit = other.logit;
    }
    if (sampling) lse_merge(best.m, best.s, other.m, other.s);
  }
  if (lane == 0) {
    cand[r] = best.idx;
    if (qs) {
      qs[r].logit = best.logit;
      qs[r].lse = sampling ? best.m + logf(best.s) : NAN;
    }
  }
}

cudaError_t launch_lm_merge(const LmRec* rec, int n_tiles, int rows, int K, float inv_T,
                            int32_t* cand, dlite_qstats* qs, cudaStream_t s) {
  const int wpb = 8;
  lm_merge_kernel<<<(rows + wpb - 1) / wpb, wpb * 32, 0, s>>>(rec, n_tiles, rows, K, inv_T, cand, qs);
  return cudaGetLastError();
}

}  // namespace dlite
