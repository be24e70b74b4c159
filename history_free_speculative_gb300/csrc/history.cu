// History-KV control of the history-cost workload: the conventional drafter
// that the history-free one is compared against keeps its own draft KV, a ring
// of the last H local key / value rows per layer and request, and attends over
// it beside the block ([P1] §"本轮临时 K/V 仍然需要计算": the draft KV of a
// conventional drafter grows with the history, M_draftKV ≈ 2 L_D H n_kv d_h b;
// [P2] §"实验：三类负载，逐项看数字", ablation: 128- and 512-token
// sliding-window KV variants). Kernels:
//   hist_fill      the synthetic history (Philox, tag 6), bit-identical to the
//                  CPU definition: four uniforms summed in fp32, centred and
//                  scaled to unit variance, rounded to bf16;
//   hist_attn      split-KV attention of one key/value head's query rows
//                  (n_q / n_kv heads x G + K local rows) over one chunk of the
//                  H cached keys followed by the m + G + K block keys:
//                  bulk-copy 3-stage ring of 64-key tiles, QK^T and PV on the
//                  bf16 tensor cores (mma.sync m16n8k16, P split into two bf16
//                  parts), online softmax in registers; writes (m, l, o) per row
//                  and key half;
//   hist_combine   merges the chunk partials into the attention output and
//                  writes the round's local rows into the ring at slots
//                  (cursor + j) mod H (after every chunk of the layer has read it);
//   hist_advance   cursor += G + K (mod H) once the last layer is done.
#include <algorithm>

#include "kernels.h"
#include "tc_device.cuh"

namespace dlite {

namespace {

constexpr uint32_t kTagHist = 6;
constexpr uint32_t kHistSeedLo = 0x00000001u, kHistSeedHi = 0x48495354u;  // key of the synthetic history
constexpr int kHistKeys = 64;   // keys per shared-memory tile
constexpr int kHistStages = 3;  // tiles in flight

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// 16-byte asynchronous copy global -> shared; src_bytes = 0 fills zeros
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_a(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t_a(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// D[16 x 8] += A[16 x 16] B[16 x 8], bf16 operands, fp32 accumulation
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------- synthetic history
__global__ void hist_fill_kernel(HistFillArgs a) {
  const size_t rows = (size_t)a.Bm * a.n_kv * a.Hx;  // described rows of one layer
  const size_t per_which = (size_t)a.L * a.rows * a.d_h;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < 2 * per_which; e += stride) {
    const int which = e >= per_which;
    size_t r = e - (which ? per_which : 0);
    const int d = (int)(r % a.d_h);
    r /= a.d_h;
    const int l = (int)(r / a.rows);
    const size_t R = r % a.rows;  // row within the layer: (b n_kv + g) Hx + t
    const int t = (int)(R % a.Hx), g = (int)((R / a.Hx) % a.n_kv), b = (int)(R / ((size_t)a.Hx * a.n_kv));
    float v = 0.f;  // the block rows past the ring, and padding, start as zeros
    if (R < rows && t < a.H) {
      const uint4 w = philox((uint32_t)t * (uint32_t)a.d_h + (uint32_t)d,
                             (uint32_t)((2 * l + which) * a.n_kv + g), (uint32_t)b, kTagHist, kHistSeedLo,
                             kHistSeedHi);
      const float acc = __fadd_rn(__fadd_rn(__fadd_rn(u01f(w.x), u01f(w.y)), u01f(w.z)), u01f(w.w));
      v = __fmul_rn(__fsub_rn(acc, 2.f), 1.7320508075688772f);  // unit variance
    }
    (which ? a.v : a.k)[e - (which ? per_which : 0)] = __float2bfloat16_rn(v);
  }
  if (a.cursor && blockIdx.x == 0)
    for (int b = threadIdx.x; b < a.Bm; b += blockDim.x) a.cursor[b] = 0;
}

// ---------------------------------------------------------------- split-KV attention over the ring
// CTA (chunk c, key/value head g, request b). The ring of (b, g) is followed in
// memory by the block's m + G + K rows (written there by the attention kernel),
// so the chunk's keys, 64-key tiles [c S, c S + S) of [ring (H) | block], are
// rows (b n_kv + g) Hx + t of one 2-D tensor: each tile is d_h / 64 TMA boxes
// of 64 rows x 128 bytes (128-byte swizzle: 16-byte chunk j of row r at j ^
// (r & 7), so ldmatrix's 8 row addresses hit distinct banks) for keys and as
// many for values, on a kHistStages ring of mbarrier-tracked stages. Rows past
// the chunk's end hold finite values (the next head's rows, or zeros past the
// tensor) and score -inf. Warp (mt, kh): query rows 16 mt .. 16 mt + 15 (row
// hh (G + K) + i = local row i of head g n_q / n_kv + hh) against key half kh
// of every tile (KS halves), with its own running max / sum / output; each
// (chunk, half) is one partial for the combine kernel.
template <int DH, int KS>
__global__ void __launch_bounds__(256) hist_attn_kernel(const __grid_constant__ CUtensorMap mk,
                                                        const __grid_constant__ CUtensorMap mv,
                                                        const HistAttnArgs a) {
  // no early trigger: this grid runs in several waves, and dependents launched
  // early would hold SM slots its later waves need
  pdl_wait();  // the queries and block rows come from the attention kernel; the ring from earlier rounds
  extern __shared__ unsigned char hsm_raw[];
  constexpr int NB = DH / 64, KW = kHistKeys / KS, NT = KW / 8, LDQ = DH + 8;
  constexpr uint32_t kBox = kHistKeys * 128, kStage = 2 * NB * kBox;  // bytes
  const uint32_t sbase = (tc::su32(hsm_raw) + 1023u) & ~1023u;       // swizzle atoms: 1 KB aligned
  unsigned char* hsm = hsm_raw + (sbase - tc::su32(hsm_raw));
  bf16* qsm = reinterpret_cast<bf16*>(hsm + kHistStages * kStage);
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nthr = blockDim.x;
  const int MT = (nthr >> 5) / KS, mt = warp % MT, kh = warp / MT;
  const int gq = lane >> 2, cq = lane & 3, mat = lane >> 3, r8 = lane & 7;
  uint64_t* full = reinterpret_cast<uint64_t*>(hsm + kHistStages * kStage + (size_t)MT * 16 * LDQ * sizeof(bf16));
  const int T = a.H + a.Tk;
  const int s0 = c * a.sub_per_chunk;
  const int ns = min(a.sub_per_chunk, (T + kHistKeys - 1) / kHistKeys - s0);
  const size_t bg = (size_t)b * a.n_kv + g;
  const int row0 = (int)(bg * a.Hx);  // tensor row of slot 0

  if (threadIdx.x == 0) {
    for (int i = 0; i < kHistStages; ++i) tc::mbar_init(tc::su32(full + i), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = threadIdx.x; i < MT * 16 * (DH / 8); i += nthr) {  // the query tile, zero padded
    const int r = i / (DH / 8), cc = i % (DH / 8);
    cp_async16(qsm + r * LDQ + cc * 8, a.q + (bg * a.QR + min(r, a.QR - 1)) * DH + cc * 8, r < a.QR ? 16 : 0);
  }
  cp_async_commit();
  __syncthreads();  // barriers initialised
  auto issue = [&](int j, int st) {  // thread 0: tile j into stage st
    const uint32_t bar = tc::su32(full + st), dst = sbase + st * kStage;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc::mbar_expect_tx(bar, kStage);
    const int y = row0 + (s0 + j) * kHistKeys;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      tc::tma_load_2d(dst + i * kBox, &mk, bar, 64 * i, y);
      tc::tma_load_2d(dst + (NB + i) * kBox, &mv, bar, 64 * i, y);
    }
  };
  if (threadIdx.x == 0)
    for (int j = 0; j < kHistStages - 1 && j < ns; ++j) issue(j, j);
  cp_async_wait<0>();
  __syncthreads();
  uint32_t qf[DH / 16][4];
#pragma unroll
  for (int kk = 0; kk < DH / 16; ++kk)
    ldsm_x4(qf[kk], qsm + (mt * 16 + (mat & 1) * 8 + r8) * LDQ + kk * 16 + (mat >> 1) * 8);

  float o[DH / 8][4];
#pragma unroll
  for (int i = 0; i < DH / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float sc = a.scale_log2;
  int j = 0;
  bool ok = true;
  for (; j < ns; ++j) {
    const int st = j % kHistStages;
    const bool got = tc::mbar_wait(tc::su32(full + st), (uint32_t)(j / kHistStages) & 1u, a.status);
    // every thread is past tile j - 1, whose stage is refilled next; tile j is in
    if (!__syncthreads_and(got)) {
      ok = false;
      break;
    }
    if (threadIdx.x == 0 && j + kHistStages - 1 < ns) issue(j + kHistStages - 1, (j + kHistStages - 1) % kHistStages);
    const int nv = min(kHistKeys, T - (s0 + j) * kHistKeys);
    const uint32_t kt = sbase + st * kStage + kh * KW * 128;  // this warp's key half
    const uint32_t vt = kt + NB * kBox;
    // S = Q K^T: 16 rows x KW keys
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk) {
      const uint32_t kaddr = kt + (kk >> 2) * kBox + ((((kk & 3) * 2 + (mat & 1)) ^ r8) << 4);
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        uint32_t bq[4];
        ldsm_x4_a(bq, kaddr + (np * 16 + (mat >> 1) * 8 + r8) * 128);
        mma_bf16(s[2 * np], qf[kk], bq[0], bq[1]);
        mma_bf16(s[2 * np + 1], qf[kk], bq[2], bq[3]);
      }
    }
    if (nv < kHistKeys) {  // keys past the end
      const int lim = nv - kh * KW;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (nt * 8 + 2 * cq + (e & 1) >= lim) s[nt][e] = -INFINITY;
    }
    // online softmax in the log2 domain: p = 2^(s c - m), m the running max of s c
    float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      x0 = fmaxf(x0, fmaxf(s[nt][0], s[nt][1]));
      x1 = fmaxf(x1, fmaxf(s[nt][2], s[nt][3]));
    }
    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 1));
    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 2));
    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 1));
    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 2));
    // a half with no valid key in this tile keeps its max (x = -inf)
    const float n0 = fmaxf(m0, x0 * sc), n1 = fmaxf(m1, x1 * sc);
    if (n0 != m0 || n1 != m1) {  // rescale only when a row's max moved
      const float al0 = n0 == m0 ? 1.f : tc::ex2_approx(m0 - n0), al1 = n1 == m1 ? 1.f : tc::ex2_approx(m1 - n1);
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int dt = 0; dt < DH / 8; ++dt) {
        o[dt][0] *= al0;
        o[dt][1] *= al0;
        o[dt][2] *= al1;
        o[dt][3] *= al1;
      }
      m0 = n0;
      m1 = n1;
    }
    // a row with no valid key yet (m = -inf) has every p = 0
    const float b0 = m0 == -INFINITY ? 0.f : -m0, b1 = m1 == -INFINITY ? 0.f : -m1;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      s[nt][0] = tc::ex2_approx(fmaf(s[nt][0], sc, b0));
      s[nt][1] = tc::ex2_approx(fmaf(s[nt][1], sc, b0));
      s[nt][2] = tc::ex2_approx(fmaf(s[nt][2], sc, b1));
      s[nt][3] = tc::ex2_approx(fmaf(s[nt][3], sc, b1));
      l0 += s[nt][0] + s[nt][1];
      l1 += s[nt][2] + s[nt][3];
    }
    // O += P V with P = hi + lo in bf16 (to ~2^-16; the score accumulators are the A fragments)
#pragma unroll
    for (int kk = 0; kk < KW / 16; ++kk) {
      const float* p0 = s[2 * kk];
      const float* p1 = s[2 * kk + 1];
      const uint32_t ah[4] = {pack2(p0[0], p0[1]), pack2(p0[2], p0[3]), pack2(p1[0], p1[1]), pack2(p1[2], p1[3])};
      float lo[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        lo[e] = p0[e] - round_bf16(p0[e]);
        lo[4 + e] = p1[e] - round_bf16(p1[e]);
      }
      const uint32_t al[4] = {pack2(lo[0], lo[1]), pack2(lo[2], lo[3]), pack2(lo[4], lo[5]), pack2(lo[6], lo[7])};
      const uint32_t vrow = vt + (kk * 16 + (mat & 1) * 8 + r8) * 128;
#pragma unroll
      for (int dp = 0; dp < DH / 16; ++dp) {
        uint32_t bv[4];
        ldsm_x4_t_a(bv, vrow + (dp >> 2) * kBox + ((((dp & 3) * 2 + (mat >> 1)) ^ r8) << 4));
        mma_bf16(o[2 * dp], ah, bv[0], bv[1]);
        mma_bf16(o[2 * dp + 1], ah, bv[2], bv[3]);
        mma_bf16(o[2 * dp], al, bv[0], bv[1]);
        mma_bf16(o[2 * dp + 1], al, bv[2], bv[3]);
      }
    }
  }
  if (!ok) {  // a copy never landed: let the issued ones finish (bounded), flag, leave
    if (threadIdx.x == 0)
      for (int k = j; k < min(ns, j + kHistStages - 1); ++k)
        tc::mbar_wait(tc::su32(full + k % kHistStages), (uint32_t)(k / kHistStages) & 1u, a.status);
    __syncthreads();
    return;
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const size_t pr = ((bg * a.nchunk + c) * KS + kh) * a.QR;  // first partial row of this warp's half
  const int q0 = mt * 16 + gq, q1 = q0 + 8;
#pragma unroll
  for (int dt = 0; dt < DH / 8; ++dt) {
    if (q0 < a.QR)
      *reinterpret_cast<float2*>(a.part_o + (pr + q0) * DH + dt * 8 + 2 * cq) = make_float2(o[dt][0], o[dt][1]);
    if (q1 < a.QR)
      *reinterpret_cast<float2*>(a.part_o + (pr + q1) * DH + dt * 8 + 2 * cq) = make_float2(o[dt][2], o[dt][3]);
  }
  if (cq == 0) {
    if (q0 < a.QR) *reinterpret_cast<float2*>(a.part_ml + (pr + q0) * 2) = make_float2(m0, l0);
    if (q1 < a.QR) *reinterpret_cast<float2*>(a.part_ml + (pr + q1) * 2) = make_float2(m1, l1);
  }
}

// ---------------------------------------------------------------- combine + ring append
// CTA (query row r, head g, request b), one thread per column: o = sum_c
// 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c, rounded to bf16 into the attention
// output; CTAs r < G + K also copy block row m + r (the round's local key /
// value rows, stored behind the ring) to ring slot (cursor + r) mod H.
__global__ void hist_combine_kernel(HistCombineArgs a) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, g = blockIdx.y, b = blockIdx.z, d = threadIdx.x;
  const size_t bg = (size_t)b * a.n_kv + g;
  const float2* ml = reinterpret_cast<const float2*>(a.part_ml) + bg * a.nchunk * a.QR + r;
  const float* po = a.part_o + (bg * a.nchunk * a.QR + r) * a.d_h + d;
  float M = -INFINITY;
  for (int c = 0; c < a.nchunk; ++c) M = fmaxf(M, ml[(size_t)c * a.QR].x);
  float L = 0.f, acc = 0.f;
  for (int c = 0; c < a.nchunk; ++c) {
    const float2 v = ml[(size_t)c * a.QR];
    const float w = exp2f(v.x - M);
    L = fmaf(w, v.y, L);
    acc = fmaf(w, po[(size_t)c * a.QR * a.d_h], acc);
  }
  const int hpg = a.n_q / a.n_kv, hh = r / a.K1, i = r % a.K1;
  a.o[((size_t)b * a.K1 + i) * a.n_q * a.d_h + (size_t)(g * hpg + hh) * a.d_h + d] = __float2bfloat16_rn(acc / L);
  if (r < a.K1) {
    const int slot = (a.cursor[b] + r) % a.H;
    const size_t src = (bg * a.Hx + a.H + a.m + r) * a.d_h + d, dst = (bg * a.Hx + slot) * a.d_h + d;
    a.kc[dst] = a.kc[src];
    a.vc[dst] = a.vc[src];
  }
}

__global__ void hist_advance_kernel(int* cursor, int B, int n, int H) {
  pdl_trigger();
  pdl_wait();
  for (int b = threadIdx.x; b < B; b += blockDim.x) cursor[b] = (cursor[b] + n) % H;
}

}  // namespace

size_t hist_attn_smem(int d_h, int QR) {  // 1 KB alignment slack, stages, query tile, barriers
  const int MT = (QR + 15) / 16;
  return 1024 + (size_t)kHistStages * 2 * kHistKeys * d_h * sizeof(bf16) + (size_t)MT * 16 * (d_h + 8) * sizeof(bf16) +
         kHistStages * sizeof(uint64_t);
}

int hist_key_splits(int QR) { return (QR + 15) / 16 <= 4 ? 2 : 1; }

HistPlan hist_plan(int B, int n_kv, int H, int Tk, int QR, int d_h, int num_sms) {
  HistPlan p;
  const int nsub = (H + Tk + kHistKeys - 1) / kHistKeys;
  const long long BG = (long long)B * n_kv;
  const size_t smem = hist_attn_smem(d_h, QR);
  const long long resident = (long long)num_sms * std::max<size_t>(1, std::min<size_t>(8, 227 * 1024 / (smem + 1024)));
  const int max_chunks = (int)std::max<long long>(1, std::min<long long>(nsub, hist_max_ctas(num_sms) / BG));
  // cost in sub-tile loads per resident slot: waves x tile loads, plus the
  // partials written and read back (fp32 rows of d_h + 2 values)
  const double part_tiles = (double)QR * (d_h + 2) * 8 / ((double)kHistKeys * d_h * 4);
  double best = 1e300;
  for (int n = 1; n <= max_chunks; ++n) {
    const int spc = (nsub + n - 1) / n, ne = (nsub + spc - 1) / spc;
    const long long waves = (BG * ne + resident - 1) / resident;
    const double cost = (double)waves * spc + (double)BG * ne * part_tiles / resident;
    if (cost < best - 1e-9) {
      best = cost;
      p.sub_per_chunk = spc;
      p.nchunk = ne;
    }
  }
  return p;
}

long long hist_max_ctas(int num_sms) { return 8LL * num_sms; }

cudaError_t launch_hist_fill(const HistFillArgs& a, cudaStream_t s) {
  const size_t n = 2 * (size_t)a.L * a.Bm * a.n_kv * a.H * a.d_h;
  const int blocks = (int)std::min<size_t>((n + 255) / 256, (size_t)device_sms() * 16);
  hist_fill_kernel<<<std::max(blocks, 1), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_hist_attn(const CUtensorMap* mk, const CUtensorMap* mv, const HistAttnArgs& a, int d_h,
                             cudaStream_t s) {
  const int MT = (a.QR + 15) / 16, KS = hist_key_splits(a.QR);
  if (MT * KS > 8 || a.nchunk < 1 || (d_h != 64 && d_h != 128)) return cudaErrorInvalidValue;
  const size_t smem = hist_attn_smem(d_h, a.QR);
  void (*fn)(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap, const HistAttnArgs) =
      d_h == 128 ? (KS == 2 ? hist_attn_kernel<128, 2> : hist_attn_kernel<128, 1>)
                 : (KS == 2 ? hist_attn_kernel<64, 2> : hist_attn_kernel<64, 1>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(fn, dim3(a.nchunk, a.n_kv, a.B), dim3(32 * MT * KS), smem, s, *mk, *mv, a);
}

cudaError_t launch_hist_combine(const HistCombineArgs& a, cudaStream_t s) {
  return launch_pdl(hist_combine_kernel, dim3(a.QR, a.n_kv, a.B), dim3(a.d_h), 0, s, a);
}

cudaError_t launch_hist_advance(int* cursor, int B, int n, int H, cudaStream_t s) {
  return launch_pdl(hist_advance_kernel, dim3(1), dim3(32), 0, s, cursor, B, n, H);
}

}  // namespace dlite
