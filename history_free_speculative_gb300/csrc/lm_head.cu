// Persistent LM-head kernel: logits = h E^T with the argmax / Gumbel-max
// selection and the log-sum-exp folded in, logits never written to memory.
//
// One CTA per SM walks the vocabulary slabs blockIdx.x, blockIdx.x + grid, ...
// (N ids each). The accumulator in TMEM is double-buffered: while the MMA warp
// accumulates slab t into one buffer, the epilogue warps score slab t-1 from
// the other, so the sampling arithmetic (Philox, two logarithms and one
// exponential per logit) runs under the stream of E from HBM instead of after
// it. Every epilogue thread owns one row of h and keeps its running top-4 and
// LSE partials over all slabs of its CTA in registers; it writes one record
// per CTA and column group at the end, which the merge kernel combines.
//
// Warp roles: warp 0 TMA producer (E slab tile + h tiles per 64-wide k block,
// through a ring of shared-memory stages), warp 1 TMEM owner and MMA issuer,
// warps 2 .. 2 + 4 * kLmGroups - 1 epilogue (warp w reads TMEM lane quadrant
// w % 4; the column groups split each slab's columns).
// Every wait is bounded (~2 s); on expiry the status word is flagged, the
// producer waits (bounded) for its own copies in flight, the MMA warp for its
// own products, and the kernel frees TMEM and returns.
#include "tc_device.cuh"
#include "tc_gemm.h"

namespace dlite {
namespace tc {

constexpr int kLmGroups = 4;
constexpr int kLmThreads = 64 + 128 * kLmGroups;

// Fold one 16-column chunk whose first nv columns are vocabulary ids (nv may
// be <= 0 past the end of the vocabulary, or exceed 16).
__device__ __forceinline__ void fold_cols(LmAcc& a, const uint32_t (&raw)[16], int v0, int nv, bool sampling,
                                          float c2s, const PhiloxRow& pr, uint32_t k0, uint32_t k1) {
  if (nv >= 16) {
    if (sampling)
      lm_fold16<true, true>(a, raw, v0, 16, c2s, pr, k0, k1);
    else
      lm_fold16<false, true>(a, raw, v0, 16, c2s, pr, k0, k1);
  } else if (nv > 0) {
    if (sampling)
      lm_fold16<true, false>(a, raw, v0, nv, c2s, pr, k0, k1);
    else
      lm_fold16<false, false>(a, raw, v0, nv, c2s, pr, k0, k1);
  }
}

template <int NMT, int N>
__global__ void __launch_bounds__(kLmThreads, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw,
                   const LmParams p) {
  constexpr uint32_t kAccCols = (uint32_t)(NMT * N);  // one accumulator buffer
  constexpr uint32_t kTmemCols = 2 * kAccCols;
  static_assert(kTmemCols <= 512, "two accumulators must fit TMEM");
  constexpr uint32_t kWTile = (uint32_t)N * 128u;     // one k block of the E slab
  constexpr int kColsPerGroup = N / kLmGroups;         // multiple of 16

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)base;
  // barriers: full[stages] empty[stages] acc_full[2] acc_empty[2] done
  const uint32_t full0 = su32(bars), empty0 = su32(bars + p.stages);
  const uint32_t accf0 = su32(bars + 2 * p.stages), acce0 = su32(bars + 2 * p.stages + 2);
  const uint32_t done = su32(bars + 2 * p.stages + 4);
  uint32_t* tmem_holder = (uint32_t*)(bars + 2 * p.stages + 5);
  uint8_t* smem = base + 1024;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool aborted = p.status && (*(volatile int*)p.status & kDevTimeout);
  const int G = (int)gridDim.x;
  const int n_mine = aborted || (int)blockIdx.x >= p.n_slabs ? 0 : (p.n_slabs - 1 - (int)blockIdx.x) / G + 1;
  const int nkb = p.kblocks;
  const int rot = (int)(blockIdx.x % (unsigned)nkb);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 4 * kLmGroups);
    }
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_trigger();

  if (warp == 0) {  // ---------------- TMA producer
    const uint32_t a_slot = a_slot_bytes(p.x_box);
    const uint32_t bytes = kWTile + (uint32_t)NMT * (uint32_t)p.x_box * 128u;
    auto load_w = [&](int slab, int j, int s) {
      const uint32_t st = su32(smem + (size_t)s * p.stage_bytes);
      const uint32_t fb = full0 + 8 * s;
      mbar_expect_tx(fb, bytes);
      tma_load_4d(st + (uint32_t)NMT * a_slot, &mw, fb, (j + rot) % nkb, slab * (N / 64));
    };
    auto load_x = [&](int j, int s) {
      const uint32_t st = su32(smem + (size_t)s * p.stage_bytes);
      const uint32_t fb = full0 + 8 * s;
      const int kx = ((j + rot) % nkb) * 64;
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) tma_load_2d(st + (uint32_t)mt * a_slot, &mx, fb, kx, mt * 128);
    };
    // E does not depend on the previous kernel: its first tiles are requested
    // before waiting for h.
    const int total = n_mine * nkb;
    const int pre = total < p.stages ? total : p.stages;
    if (lane == 0)
      for (int i = 0; i < pre; ++i) load_w((int)blockIdx.x + (i / nkb) * G, i % nkb, i);
    __syncwarp();
    pdl_wait();
    if (lane == 0)
      for (int i = 0; i < pre; ++i) load_x(i % nkb, i);
    __syncwarp();
    int issued = pre;
    bool ok = true;
    for (int i = pre; i < total; ++i) {
      const int s = i % p.stages;
      if (!mbar_wait_warp(empty0 + 8 * s, (uint32_t)(i / p.stages - 1) & 1, p.status)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        load_w((int)blockIdx.x + (i / nkb) * G, i % nkb, s);
        load_x(i % nkb, s);
      }
      __syncwarp();
      issued = i + 1;
    }
    if (!ok) {  // let the copies still in flight land before the CTA exits
      for (int i = issued - p.stages < 0 ? 0 : issued - p.stages; i < issued; ++i)
        mbar_wait_warp(full0 + 8 * (i % p.stages), (uint32_t)(i / p.stages) & 1, nullptr);
    }
  } else if (warp == 1) {  // ---------------- MMA issuer
    const uint32_t idesc = idesc_bf16(128, N);
    const uint32_t a_slot = a_slot_bytes(p.x_box);
    const uint64_t aslot = (uint64_t)(a_slot >> 4);
    const uint64_t wbase = (uint64_t)(((uint32_t)NMT * a_slot) >> 4);
    const uint64_t desc0 = sw128_desc(su32(smem));
    const uint64_t sdelta = (uint64_t)(p.stage_bytes >> 4);
    int i = 0;
    bool ok = true;
    for (int t = 0; t < n_mine && ok; ++t) {
      const int b = t & 1;
      if (t >= 2 && !mbar_wait_warp(acce0 + 8 * b, (uint32_t)((t >> 1) - 1) & 1, p.status)) break;
      fence_after();
      const uint32_t dbase = tmem + (uint32_t)b * kAccCols;
      for (int j = 0; j < nkb; ++j, ++i) {
        const int s = i % p.stages;
        if (!mbar_wait_warp(full0 + 8 * s, (uint32_t)(i / p.stages) & 1, p.status)) {
          ok = false;
          break;
        }
        fence_after();
        if (lane == 0) {
          const uint64_t a0 = desc0 + sdelta * (uint64_t)s;
          const uint64_t b0 = a0 + wbase;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int mt = 0; mt < NMT; ++mt)
              umma_bf16(dbase + (uint32_t)(mt * N), a0 + (uint64_t)(kk * 2) + (uint64_t)mt * aslot,
                        b0 + (uint64_t)(kk * 2), idesc, (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(empty0 + 8 * s);
        }
        __syncwarp();
      }
      if (ok && lane == 0) umma_commit(accf0 + 8 * b);
      __syncwarp();
    }
    // every product issued has finished before TMEM is released
    if (lane == 0) umma_commit(done);
    __syncwarp();
    mbar_wait_warp(done, 0, nullptr);
  } else {  // ---------------- epilogue warps
    const int q = warp & 3;
    const int eg = (warp - 2) >> 2;
    const int c_lo = eg * kColsPerGroup;
    const bool sampling = p.inv_T > 0.f;
    const float c2s = p.inv_T * kLog2e;
    pdl_wait();  // positions are read below; records are written at the end
    LmAcc acc[NMT];
    PhiloxRow pr[NMT];
    int row[NMT];
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt) {
      lm_acc_init(acc[mt]);
      row[mt] = mt * 128 + q * 32 + lane;
      pr[mt] = {0u, 0u, 0u};
      if (sampling && row[mt] < p.rows) {
        const int req = row[mt] / p.K_draft;
        const uint32_t pos = (uint32_t)(p.pos[req] + (row[mt] % p.K_draft) + 1);
        pr[mt] = philox_row_init(pos, (uint32_t)req, kTagGumbel, p.k0, p.k1);
      }
    }
    for (int t = 0; t < n_mine; ++t) {
      const int b = t & 1;
      const int slab = (int)blockIdx.x + t * G;
      if (!mbar_wait_warp(accf0 + 8 * b, (uint32_t)(t >> 1) & 1, p.status)) break;
      fence_after();
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) {
        const uint32_t tbase =
            tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)b * kAccCols + (uint32_t)(mt * N + c_lo);
        const bool valid = row[mt] < p.rows;
        if constexpr (kColsPerGroup % 32 == 0) {
#pragma unroll
          for (int c = 0; c < kColsPerGroup; c += 32) {
            uint32_t r0[16], r1[16];
            tmem_ld16_nowait(tbase + c, r0);
            tmem_ld16_nowait(tbase + c + 16, r1);
            tmem_wait_ld();
            const int v0 = slab * N + c_lo + c;
            if (valid) {
              fold_cols(acc[mt], r0, v0, p.outs - v0, sampling, c2s, pr[mt], p.k0, p.k1);
              fold_cols(acc[mt], r1, v0 + 16, p.outs - v0 - 16, sampling, c2s, pr[mt], p.k0, p.k1);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < kColsPerGroup; c += 16) {
            uint32_t r0[16];
            tmem_ld16_nowait(tbase + c, r0);
            tmem_wait_ld();
            const int v0 = slab * N + c_lo + c;
            if (valid) fold_cols(acc[mt], r0, v0, p.outs - v0, sampling, c2s, pr[mt], p.k0, p.k1);
          }
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce0 + 8 * b);
    }
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt)
      if (row[mt] < p.rows)
        lm_acc_store(acc[mt], p.rec + ((size_t)blockIdx.x * kLmGroups + eg) * p.rows + row[mt]);
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------- host side

LmPlan lm_plan_persistent(int rows, int outs, int K, int num_sms) {
  LmPlan pl;
  if (rows < 1 || rows > 256 || K % 64 || K < 64 || outs < 8 || num_sms < 1) return pl;
  pl.n_mt = rows > 128 ? 2 : 1;
  pl.N = pl.n_mt == 2 ? 128 : 256;
  const int nmax_out = ((outs + 63) / 64) * 64;  // tiled E rows
  while (pl.N > 64 && pl.N > nmax_out) pl.N >>= 1;
  pl.x_box = x_box_rows(rows);
  pl.kblocks = K / 64;
  pl.stage_bytes = (uint32_t)pl.N * 128u + (uint32_t)pl.n_mt * a_slot_bytes(pl.x_box);
  int stages = (int)((kSmemBudget - 2048 - kTailPad) / pl.stage_bytes);
  if (stages > 8) stages = 8;
  if (stages < 2) return pl;
  pl.stages = stages;
  pl.n_slabs = (outs + pl.N - 1) / pl.N;
  pl.grid = pl.n_slabs < num_sms ? pl.n_slabs : num_sms;
  pl.groups = kLmGroups;
  pl.ok = true;
  return pl;
}

size_t lm_smem_bytes(const LmPlan& pl) {
  return 1024 /* align */ + 1024 /* barriers */ + (size_t)pl.stages * pl.stage_bytes + kTailPad;
}

typedef void (*LmKernelFn)(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap,
                           const LmParams);

static LmKernelFn lm_pick(int nmt, int N) {
  if (nmt == 1 && N == 256) return lm_head_kernel<1, 256>;
  if (nmt == 1 && N == 128) return lm_head_kernel<1, 128>;
  if (nmt == 1 && N == 64) return lm_head_kernel<1, 64>;
  if (nmt == 2 && N == 128) return lm_head_kernel<2, 128>;
  if (nmt == 2 && N == 64) return lm_head_kernel<2, 64>;
  return nullptr;
}

cudaError_t launch_lm_persistent(const LmPlan& pl, const CUtensorMap* x, const CUtensorMap* w, LmParams prm,
                                 cudaStream_t s) {
  LmKernelFn fn = lm_pick(pl.n_mt, pl.N);
  if (!fn || !pl.ok) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
  if (e != cudaSuccess) return e;
  prm.n_slabs = pl.n_slabs;
  prm.kblocks = pl.kblocks;
  prm.stages = pl.stages;
  prm.stage_bytes = pl.stage_bytes;
  prm.x_box = pl.x_box;
  return launch_pdl(fn, dim3(pl.grid), dim3(kLmThreads), lm_smem_bytes(pl), s, *x, *w, prm);
}

}  // namespace tc
}  // namespace dlite
