// Persistent LM-head kernel: logits = h E^T with the argmax / the first level
// of the two-level draw (chunk Gumbel-max) and the log-sum-exp folded in;
// logits never reach memory.
//
// Up to 128 rows of h: one CTA per SM walks the vocabulary slabs blockIdx.x,
// blockIdx.x + grid, ... (N = 256 ids each) with one M = 128 MMA per 16-wide k
// step. 129..256 rows: clusters of two CTAs (CTA pairs) walk the slabs with
// 2-SM MMAs (tcgen05.mma.cta_group::2, M = 256): rank c holds rows 128c.. of h
// and E rows 128c.. of each 256-id slab, so every SM streams half a slab per
// step and reads 8 KB of operands per 16-wide k step from shared memory (a
// 128 x 256 MMA on one SM reads 12 KB, more than shared memory delivers at the
// tensor pipe's rate once the TMA writes are added). In both modes the
// accumulator is double-buffered in TMEM (2 x 256 columns): while slab t
// accumulates, the epilogue warps score slab t-1, so the sampling arithmetic
// runs under the stream of E from HBM. Every epilogue thread owns one row and
// keeps its running top-4 and LSE partials over all slabs of its CTA in
// registers; at the end the column groups of a row are combined in shared
// memory and one record per walk is written; the merge kernel combines them.
//
// With at most 32 rows and a short k extent (the gated head's per-step W_o
// product: 8 k blocks per slab) scoring, not the E stream, paces a slab, and
// rows 0..31 sit in TMEM lane quadrant 0, which only the warps of one SM
// sub-partition can read. Then (`rep`) the h tile is loaded four times, at
// rows 0, 32, 64 and 96, so every quadrant holds the same logits, and the
// warp of quadrant q scores a quarter of its column group: four times the
// epilogue warps, a quarter of the columns each.
//
// Warp roles: warp 0 TMA producer (E slab k block + h tile per 64-wide k
// block, through a ring of shared-memory stages; in a pair every copy signals
// rank 0's barrier), warp 1 TMEM owner and MMA issuer (rank 0 of a pair),
// warps 2 .. 2 + 4 * kLmGroups - 1 epilogue (warp w reads TMEM lane quadrant
// w % 4; the column groups split each slab's columns).
// Every wait is bounded (~2 s); on expiry the status word is flagged, the
// roles run to the end and the kernel frees TMEM and returns.
#include "tc_device.cuh"
#include "tc_gemm.h"

namespace dlite {
namespace tc {

constexpr int kLmGroups = 4;
constexpr int kLmThreads = 64 + 128 * kLmGroups;

// Fold one 16-column chunk whose first nv columns are vocabulary ids (nv may
// exceed 16). Warp-collective; `active` is this lane's row validity.
__device__ __forceinline__ void fold_cols(LmAcc& a, const uint32_t (&raw)[16], int v0, int nv, bool sampling,
                                          float c2s, const PhiloxRow& pr, uint32_t k0, uint32_t k1,
                                          bool active) {
  if (nv >= 16) {
    if (sampling)
      lm_fold16<true, true>(a, raw, v0, 16, c2s, pr, k0, k1, active);
    else
      lm_fold16<false, true>(a, raw, v0, 16, c2s, pr, k0, k1, active);
  } else if (nv > 0) {
    if (sampling)
      lm_fold16<true, false>(a, raw, v0, nv, c2s, pr, k0, k1, active);
    else
      lm_fold16<false, false>(a, raw, v0, nv, c2s, pr, k0, k1, active);
  }
}

template <int N, bool PAIR>
__global__ void __launch_bounds__(kLmThreads, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap mx0, const __grid_constant__ CUtensorMap mx1,
                   const __grid_constant__ CUtensorMap mw, const LmParams p) {
  constexpr uint32_t kAccCols = (uint32_t)N;  // one accumulator buffer
  constexpr uint32_t kTmemCols = 2 * kAccCols;
  static_assert(kTmemCols <= 512, "two accumulators must fit TMEM");
  constexpr uint32_t kWRows = PAIR ? N / 2 : N;      // E rows of a slab in this CTA
  constexpr uint32_t kWTile = kWRows * 128u;        // one k block of them
  constexpr int kColsPerGroup = N / kLmGroups;      // multiple of 16

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
  // walk geometry: unit = index of the slab walk, tile = 128-row tile of h
  const int tile = PAIR ? (int)cluster_rank() : 0;
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int n_units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int x_box = tile ? p.x_box1 : p.x_box0;
  const int n_mine = aborted || unit >= p.n_slabs ? 0 : (p.n_slabs - 1 - unit) / n_units + 1;
  const int nkb = p.kblocks;
  const int rot = unit % nkb;  // the same k order in both CTAs of a pair

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, (PAIR ? 2 : 1) * 4 * kLmGroups);  // every epilogue warp (of both CTAs)
    }
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    if (PAIR) {  // one warp of each CTA allocates the pair's columns together
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_holder)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_holder)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();  // both CTAs' barriers exist before any copy, commit or arrival
  fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_trigger();

  if (warp == 0) {  // ---------------- TMA producer
    // stage: [h tile: x_box rows in a slot of x_box0 rows][E slab k block: kWRows rows]
    const uint32_t wofs = a_slot_bytes(p.rep ? 128 : p.x_box0);
    // bytes landing per stage: in a pair, rank 0's barrier counts both CTAs' copies
    const uint32_t bytes = PAIR ? 2u * kWTile + (uint32_t)(p.x_box0 + p.x_box1) * 128u
                                : kWTile + (uint32_t)x_box * 128u * (p.rep ? 4u : 1u);
    const uint32_t fullb = PAIR ? map_to_rank(full0, 0) : full0;
    const CUtensorMap* mx = tile ? &mx1 : &mx0;
    // One lane issues every copy, so its per-stage instruction latency bounds
    // the stream: the stage, its phase, the k block and the slab advance by
    // increments (integer division by a runtime divisor costs tens of cycles).
    auto load_w = [&](int s, int kb, int slab) {
      const uint32_t st = su32(smem + (size_t)s * p.stage_bytes);
      if (!PAIR || tile == 0) mbar_expect_tx(full0 + 8 * s, bytes);
      const int wrow = (slab * N + tile * (int)kWRows) >> 6;
      if (PAIR)
        tma_load_4d_pair(st + wofs, &mw, fullb + 8 * s, kb, wrow);
      else
        tma_load_4d(st + wofs, &mw, fullb + 8 * s, kb, wrow);
    };
    auto load_x = [&](int s, int kb) {
      const uint32_t st = su32(smem + (size_t)s * p.stage_bytes);
      const int kx = kb * 64;
      if (PAIR)
        tma_load_2d_pair(st, mx, fullb + 8 * s, kx, tile * 128);
      else if (p.rep)  // one copy of the rows per TMEM lane quadrant
        for (int q4 = 0; q4 < 4; ++q4) tma_load_2d(st + q4 * 32 * 128, mx, fullb + 8 * s, kx, 0);
      else
        tma_load_2d(st, mx, fullb + 8 * s, kx, tile * 128);
    };
    // E does not depend on the previous kernel: its first tiles are requested
    // before waiting for h.
    const int total = n_mine * nkb;
    const int pre = total < p.stages ? total : p.stages;
    if (lane == 0) {
      int kb = rot, j = 0, slab = unit;
      for (int i = 0; i < pre; ++i) {
        load_w(i, kb, slab);
        if (++kb == nkb) kb = 0;
        if (++j == nkb) {
          j = 0;
          slab += n_units;
        }
      }
    }
    __syncwarp();
    pdl_wait();
    if (lane == 0) {
      int kb = rot;
      for (int i = 0; i < pre; ++i) {
        load_x(i, kb);
        if (++kb == nkb) kb = 0;
      }
    }
    __syncwarp();
    // cursor of copy i = pre: stage s (phase ph of its use), k block kb, the
    // j-th block of the slab
    int s = pre % p.stages, j = pre % nkb;
    int kb = (j + rot) % nkb, slab = unit + (pre / nkb) * n_units;
    uint32_t ph = (uint32_t)(pre / p.stages) & 1u;
    int issued = pre;
    bool ok = true;
    for (int i = pre; i < total; ++i) {
      // the slot's previous use (copy i - stages) had the other phase
      if (!mbar_wait_warp(empty0 + 8 * s, ph ^ 1u, p.status)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        load_w(s, kb, slab);
        load_x(s, kb);
      }
      __syncwarp();
      issued = i + 1;
      if (++s == p.stages) {
        s = 0;
        ph ^= 1u;
      }
      if (++kb == nkb) kb = 0;
      if (++j == nkb) {
        j = 0;
        slab += n_units;
      }
    }
    if (!ok && (!PAIR || tile == 0)) {  // let the copies still in flight land before the CTA exits
      for (int i = issued - p.stages < 0 ? 0 : issued - p.stages; i < issued; ++i)
        mbar_wait_warp(full0 + 8 * (i % p.stages), (uint32_t)(i / p.stages) & 1, nullptr);
    }
  } else if (warp == 1) {  // ---------------- MMA issuer (rank 0 of a pair)
    if (PAIR && tile != 0) goto mma_done;
    {
    const uint32_t idesc = idesc_bf16(PAIR ? 256 : 128, N);
    const uint64_t wbase = (uint64_t)(a_slot_bytes(p.rep ? 128 : p.x_box0) >> 4);
    const uint64_t desc0 = sw128_desc(su32(smem));
    const uint64_t sdelta = (uint64_t)(p.stage_bytes >> 4);
    int s = 0;  // stage of the next k block and the phase of its use
    uint32_t ph = 0;
    bool ok = true;
    for (int t = 0; t < n_mine && ok; ++t) {
      const int b = t & 1;
      if (t >= 2 && !mbar_wait_warp(acce0 + 8 * b, (uint32_t)((t >> 1) - 1) & 1, p.status)) break;
      fence_after();
      const uint32_t dcol = tmem + (uint32_t)b * kAccCols;
      for (int j = 0; j < nkb; ++j) {
        if (!mbar_wait_warp(full0 + 8 * s, ph, p.status)) {
          ok = false;
          break;
        }
        fence_after();
        if (lane == 0) {
          const uint64_t a0 = desc0 + sdelta * (uint64_t)s;
          const uint64_t b0 = a0 + wbase;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // +32 B along K = +2 in the encoded start address
            if (PAIR)
              umma_bf16_pair(dcol, a0 + (uint64_t)(kk * 2), b0 + (uint64_t)(kk * 2), idesc,
                             (j > 0 || kk > 0) ? 1u : 0u);
            else
              umma_bf16(dcol, a0 + (uint64_t)(kk * 2), b0 + (uint64_t)(kk * 2), idesc,
                        (j > 0 || kk > 0) ? 1u : 0u);
          }
          if (PAIR)
            umma_commit_pair(empty0 + 8 * s);
          else
            umma_commit(empty0 + 8 * s);
        }
        __syncwarp();
        if (++s == p.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (ok && lane == 0) {
        if (PAIR)
          umma_commit_pair(accf0 + 8 * b);
        else
          umma_commit(accf0 + 8 * b);
      }
      __syncwarp();
    }
    // every product issued has finished before TMEM is released
    if (lane == 0) {
      if (PAIR)
        umma_commit_pair(done);
      else
        umma_commit(done);
    }
    __syncwarp();
    mbar_wait_warp(done, 0, nullptr);
    }
  mma_done:;
  } else {  // ---------------- epilogue warps
    const int q = warp & 3;
    const int eg = (warp - 2) >> 2;
    const bool rep = !PAIR && p.rep && kColsPerGroup == 64;
    const int width = rep ? kColsPerGroup / 4 : kColsPerGroup;  // columns this warp scores per slab
    const int c_lo = eg * kColsPerGroup + (rep ? q * width : 0);
    const bool sampling = p.inv_T > 0.f;
    const float c2s = p.inv_T * kLog2e;
    pdl_wait();  // positions are read below; records are written at the end
    const int row = rep ? lane : tile * 128 + q * 32 + lane;
    const bool valid = row < p.rows;
    LmAcc acc;
    lm_acc_init(acc);
    PhiloxRow pr = {0u, 0u, 0u};
    if (sampling && valid) {
      const int req = row / p.K_draft;
      const uint32_t pos = (uint32_t)(p.pos[req] + (row % p.K_draft) + 1);
      pr = philox_row_init(pos, (uint32_t)req, kTagGumbel, p.k0, p.k1);
    }
    // a warp whose 32 rows are all past the end (the last tile of h) only
    // keeps the barrier protocol
    const bool any_valid = __any_sync(0xffffffffu, valid);
    const uint32_t acce_b = PAIR ? map_to_rank(acce0, 0) : acce0;
    for (int t = 0; t < n_mine; ++t) {
      const int b = t & 1;
      const int slab = unit + t * n_units;
      if (!mbar_wait_warp(accf0 + 8 * b, (uint32_t)(t >> 1) & 1, p.status)) break;
      fence_after();
      if (any_valid) {
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)b * kAccCols + (uint32_t)c_lo;
        if (rep) {  // one 16-column chunk
          uint32_t r0[16];
          tmem_ld16_nowait(tbase, r0);
          tmem_wait_ld();
          const int v0 = slab * N + c_lo;
          fold_cols(acc, r0, v0, p.outs - v0, sampling, c2s, pr, p.k0, p.k1, valid);
        } else if constexpr (kColsPerGroup % 32 == 0) {
#pragma unroll 1
          for (int c = 0; c < kColsPerGroup; c += 32) {
            uint32_t r0[16], r1[16];
            tmem_ld16_nowait(tbase + c, r0);
            tmem_ld16_nowait(tbase + c + 16, r1);
            tmem_wait_ld();
            const int v0 = slab * N + c_lo + c;
            fold_cols(acc, r0, v0, p.outs - v0, sampling, c2s, pr, p.k0, p.k1, valid);
            fold_cols(acc, r1, v0 + 16, p.outs - v0 - 16, sampling, c2s, pr, p.k0, p.k1, valid);
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < kColsPerGroup; c += 16) {
            uint32_t r0[16];
            tmem_ld16_nowait(tbase + c, r0);
            tmem_wait_ld();
            const int v0 = slab * N + c_lo + c;
            fold_cols(acc, r0, v0, p.outs - v0, sampling, c2s, pr, p.k0, p.k1, valid);
          }
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(acce_b + 8 * b)
                       : "memory");
        else
          mbar_arrive(acce0 + 8 * b);
      }
    }
    // combine the column groups of each row in shared memory (the stage memory
    // is idle once every product has completed): one record per row and walk
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    LmRec* sm_rec = reinterpret_cast<LmRec*>(smem);  // [kLmGroups][128]
    const int rl = q * 32 + lane;
    lm_acc_store(acc, sm_rec + eg * 128 + rl);
    asm volatile("bar.sync 1, %0;" ::"r"(4 * kLmGroups * 32) : "memory");  // the epilogue warps only
    if (eg == 0 && valid && (!rep || q == 0)) {
      for (int g2 = 1; g2 < kLmGroups * (rep ? 4 : 1); ++g2) {  // rep: every (group, quadrant) of the row
        const LmRec o = sm_rec[rep ? (g2 % kLmGroups) * 128 + (g2 / kLmGroups) * 32 + lane : g2 * 128 + rl];
#pragma unroll
        for (int k = 0; k < kTopK; ++k) topk_insert(acc.sc, acc.id, o.sc[k], o.id[k]);
        if (o.m != -INFINITY) {  // base-2 LSE partials
          if (acc.m == -INFINITY) {
            acc.m = o.m;
            acc.s = o.s;
          } else {
            const float mm = fmaxf(acc.m, o.m);
            acc.s = acc.s * ex2_approx(acc.m - mm) + o.s * ex2_approx(o.m - mm);
            acc.m = mm;
          }
        }
      }
      lm_acc_store(acc, p.rec + (size_t)unit * p.rows + row);
    }
  }
  fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();  // no copy, commit, arrival or MMA of the pair is outstanding past here
  if (warp == 1) {
    fence_after();
    if (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                   : "memory");
  }
}

// ---------------------------------------------------------------- host side

LmPlan lm_plan_persistent(int rows, int outs, int K, int num_sms) {
  LmPlan pl;
  if (rows < 1 || rows > 256 || K % 64 || K < 64 || outs < 8 || num_sms < 2) return pl;
  pl.paired = rows > 128;
  pl.N = 256;
  const int nmax_out = ((outs + 63) / 64) * 64;  // tiled E rows
  while (pl.N > (pl.paired ? 128 : 64) && pl.N > nmax_out) pl.N >>= 1;
  if (pl.N > nmax_out && !pl.paired) return pl;
  // h tiles hold only the valid rows (rounded to 8); the 128-row MMA operand of
  // a short tile overhangs into the E tile behind it (stale bytes feeding
  // unused TMEM lanes), which needs a tail pad after the last stage only when
  // that E tile is shorter than the overhang. A pair's slots are 128 rows.
  pl.x_box0 = rows >= 128 ? 128 : (rows + 7) / 8 * 8;
  pl.x_box1 = pl.paired ? (rows - 128 + 7) / 8 * 8 : 0;
  pl.kblocks = K / 64;
  pl.rep = !pl.paired && rows <= 32 && pl.N == 256 && pl.kblocks <= 16;
  const uint32_t wrows = pl.paired ? (uint32_t)pl.N / 2 : (uint32_t)pl.N;
  pl.stage_bytes = wrows * 128u + a_slot_bytes(pl.rep ? 128 : pl.x_box0);  // rep: four 32-row copies
  pl.tail_pad = !pl.paired && !pl.rep && (uint32_t)(128 - pl.x_box0) * 128u > wrows * 128u ? kTailPad : 0;
  int stages = (int)((kSmemBudget - 2048 - pl.tail_pad) / pl.stage_bytes);
  if (stages > 8) stages = 8;
  if (stages < 2) return pl;
  pl.stages = stages;
  pl.n_slabs = (outs + pl.N - 1) / pl.N;
  const int units = pl.paired ? num_sms / 2 : num_sms;
  pl.n_units = pl.n_slabs < units ? pl.n_slabs : units;
  pl.grid = pl.paired ? 2 * pl.n_units : pl.n_units;
  pl.groups = kLmGroups;
  pl.ok = true;
  return pl;
}

size_t lm_smem_bytes(const LmPlan& pl) {
  return 1024 /* align */ + 1024 /* barriers */ + (size_t)pl.stages * pl.stage_bytes + pl.tail_pad;
}

typedef void (*LmKernelFn)(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap,
                           const __grid_constant__ CUtensorMap, const LmParams);

static LmKernelFn lm_pick(int N, bool pair) {
  if (pair) {
    if (N == 256) return lm_head_kernel<256, true>;
    if (N == 128) return lm_head_kernel<128, true>;
    return nullptr;
  }
  if (N == 256) return lm_head_kernel<256, false>;
  if (N == 128) return lm_head_kernel<128, false>;
  if (N == 64) return lm_head_kernel<64, false>;
  return nullptr;
}

cudaError_t launch_lm_persistent(const LmPlan& pl, const CUtensorMap* x0, const CUtensorMap* x1,
                                 const CUtensorMap* w, LmParams prm, cudaStream_t s) {
  LmKernelFn fn = lm_pick(pl.N, pl.paired);
  if (!fn || !pl.ok) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
  if (e != cudaSuccess) return e;
  prm.n_slabs = pl.n_slabs;
  prm.kblocks = pl.kblocks;
  prm.stages = pl.stages;
  prm.stage_bytes = pl.stage_bytes;
  prm.x_box0 = pl.x_box0;
  prm.x_box1 = pl.x_box1;
  prm.paired = pl.paired ? 1 : 0;
  prm.rep = pl.rep ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(kLmThreads);
  cfg.dynamicSmemBytes = lm_smem_bytes(pl);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pl.paired ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, fn, *x0, x1 ? *x1 : *x0, *w, prm);
}

}  // namespace tc
}  // namespace dlite
