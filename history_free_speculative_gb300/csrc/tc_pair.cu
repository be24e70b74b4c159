// Tensor-core GEMM on CTA pairs (2-SM MMA), persistent and stream-K, for the
// bf16 products with more than 128 activation rows:
//
//   part[z][r][o]: the product X[r, :] . W[o, :] is the sum over the planes z
//   that the split descriptor (Splits, internal.h) gives for (r, o).
//
// A cluster of two CTAs computes 256-row x 256-column tiles with
// tcgen05.mma.cta_group::2 (M = 256): CTA rank c holds rows 128c .. 128c+127 of
// the tile's rows of X and weight rows 128c .. 128c+127 of its output slab in
// its own shared memory; each CTA's TMEM receives its 128 rows over all 256
// columns. Per SM and 16-wide k step the MMA reads 8 KB of operands (half of
// what a 128 x 256 MMA on one SM reads), so it runs at the tensor pipe's rate.
//
// The work is U = tiles x k blocks units in tile-major order; pair p takes the
// contiguous units [p U / G, (p + 1) U / G), i.e. a piece of one or more tiles,
// so every SM gets the same number of k blocks whatever the shape. Each piece
// (segment) accumulates in one of two TMEM buffers; its epilogue writes the
// fp32 partial of its 256 x 256 block to plane (p - first worker of the tile)
// while the MMAs of the next segment run in the other buffer.
//
// Warp roles per CTA: warp 0 TMA producer (both CTAs; every copy signals rank
// 0's full barrier), warp 1 TMEM owner and (rank 0 only) MMA issuer, warps
// 2-9 epilogue (warp w reads TMEM lane quadrant w % 4). Every wait is bounded
// (~2 s of %globaltimer); on expiry the status word is flagged and the roles
// run to the end instead of hanging.
#include "tc_device.cuh"
#include "tc_gemm.h"

namespace dlite {
namespace tc {

constexpr uint32_t kATile = 128 * 128;       // one 128-row x 64-k bf16 tile (16 KB)
constexpr int kPairN = 256;                  // output columns per tile
constexpr uint32_t kPairStage = 2 * kATile;  // this CTA's X tile + W tile per k block
constexpr uint32_t kPairStaging = 0;  // the epilogue stores from registers: no staging area

struct Segment {
  int tile, kb_lo, n, plane, slab, group;
};
// Next segment of the unit range [u, end) of worker `pair`: the units up to the
// end of the current tile; plane = pair - (worker owning the tile's first unit).
__device__ __forceinline__ bool next_segment(const PairParams& p, long long& u, long long end, int pair,
                                             Segment& sg) {
  if (u >= end) return false;
  const long long tile = u / p.kblocks;
  sg.tile = (int)tile;
  sg.kb_lo = (int)(u - tile * p.kblocks);
  const long long lim = (tile + 1) * p.kblocks < end ? (tile + 1) * p.kblocks : end;
  sg.n = (int)(lim - u);
  sg.plane = pair - (int)(((tile * p.kblocks + 1) * p.G - 1) / p.U);
  sg.slab = sg.tile % p.slabs;
  sg.group = sg.tile / p.slabs;
  u = lim;
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
    tc_pair_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw,
                   const PairParams p) {
  // Shared memory: [barriers | pad to 1 KB] [stage 0] ... [stage S-1] [epilogue staging]
  // stage = [X tile][W tile]; staging = 32 x 32 floats per epilogue warp
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
  const uint32_t rank = cluster_rank();
  const bool aborted = p.status && (*(volatile int*)p.status & kDevTimeout);
  const int pair = (int)(blockIdx.x >> 1);
  const long long u_begin = aborted ? 0 : (long long)pair * p.U / p.G;
  const long long u_end = aborted ? 0 : (long long)(pair + 1) * p.U / p.G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 2 * 4 * kEpiGroups);  // every epilogue warp of both CTAs
    }
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // one warp of each CTA allocates the pair's columns together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_holder)),
                 "r"(2 * kPairN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any copy, commit or arrival reaches them
  fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_trigger();

  if (warp == 0) {  // ---------------- TMA producer (both CTAs)
    const uint32_t full_leader = map_to_rank(full0, 0);
    // One lane issues every copy, so its per-stage instruction latency bounds
    // the stream: the stage and its phase advance by increments (integer
    // division by a runtime divisor costs tens of cycles).
    auto load = [&](const Segment& sg, int j, int s, bool weights, bool acts) {
      const uint32_t st = su32(smem + (size_t)s * kPairStage);
      const int kb = sg.kb_lo + j;
      if (weights) {
        if (rank == 0) mbar_expect_tx(full0 + 8 * s, 2u * kPairStage);
        tma_load_4d_pair(st + kATile, &mw, full_leader + 8 * s, kb, (sg.slab * kPairN + (int)rank * 128) >> 6);
      }
      if (acts) tma_load_2d_pair(st, &mx, full_leader + 8 * s, kb * 64, sg.group * 256 + (int)rank * 128);
    };
    // weights do not depend on the previous kernel: request the first stages'
    // weight tiles before waiting for it, then their activation tiles
    {
      long long u = u_begin;
      Segment sg;
      int i = 0;
      while (i < p.stages && next_segment(p, u, u_end, pair, sg))
        for (int j = 0; j < sg.n && i < p.stages; ++j, ++i)
          if (lane == 0) load(sg, j, i, true, false);
      __syncwarp();
      pdl_wait();
      u = u_begin;
      i = 0;
      while (i < p.stages && next_segment(p, u, u_end, pair, sg))
        for (int j = 0; j < sg.n && i < p.stages; ++j, ++i)
          if (lane == 0) load(sg, j, i, false, true);
      __syncwarp();
    }
    long long u = u_begin;
    Segment sg;
    int i = 0, s = 0;  // copy i goes to stage s in the phase ph of its use
    uint32_t ph = 0;
    bool ok = true;
    while (ok && next_segment(p, u, u_end, pair, sg)) {
      for (int j = 0; j < sg.n; ++j, ++i) {
        if (i >= p.stages) {  // the first stages were issued above
          // the slot's previous use (copy i - stages) had the other phase
          if (!mbar_wait_warp(empty0 + 8 * s, ph ^ 1u, p.status)) {
            ok = false;
            break;
          }
          if (lane == 0) load(sg, j, s, true, true);
          __syncwarp();
        }
        if (++s == p.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {  // ---------------- MMA issuer (rank 0)
    if (rank == 0) {
      const uint32_t idesc = idesc_bf16(256, kPairN);
      const uint64_t desc0 = sw128_desc(su32(smem));
      const uint64_t sdelta = (uint64_t)(kPairStage >> 4);
      const uint64_t wofs = (uint64_t)(kATile >> 4);
      long long u = u_begin;
      Segment sg;
      int t = 0, s = 0;  // stage of the next k block and the phase of its use
      uint32_t ph = 0;
      bool ok = true;
      while (ok && next_segment(p, u, u_end, pair, sg)) {
        const int b = t & 1;
        if (t >= 2 && !mbar_wait_warp(acce0 + 8 * b, (uint32_t)((t >> 1) - 1) & 1, p.status)) break;
        fence_after();
        const uint32_t dcol = tmem + (uint32_t)b * kPairN;
        for (int j = 0; j < sg.n; ++j) {
          if (!mbar_wait_warp(full0 + 8 * s, ph, p.status)) {
            ok = false;
            break;
          }
          fence_after();
          if (lane == 0) {
            const uint64_t a0 = desc0 + sdelta * (uint64_t)s;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // +32 B along K = +2 in the encoded start address
              umma_bf16_pair(dcol, a0 + (uint64_t)(kk * 2), a0 + wofs + (uint64_t)(kk * 2), idesc,
                             (j > 0 || kk > 0) ? 1u : 0u);
            umma_commit_pair(empty0 + 8 * s);
          }
          __syncwarp();
          if (++s == p.stages) {
            s = 0;
            ph ^= 1u;
          }
        }
        // also after an expired wait, so that both epilogues run to the end
        if (lane == 0) umma_commit_pair(accf0 + 8 * b);
        __syncwarp();
        ++t;
      }
      // every product issued has finished before the pair's TMEM is released
      if (lane == 0) umma_commit_pair(done);
      __syncwarp();
      mbar_wait_warp(done, 0, nullptr);
    }
  } else {  // ---------------- epilogue warps 2 .. 9 (both CTAs)
    const int q = warp & 3;
    const int eg = (warp - 2) >> 2;
    const int ncol = kPairN / kEpiGroups;
    const int c_lo = eg * ncol;
    const uint32_t acce_leader = map_to_rank(acce0, 0);
    pdl_wait();  // the partial buffer may still be read by the previous kernel
    long long u = u_begin;
    Segment sg;
    int t = 0;
    while (next_segment(p, u, u_end, pair, sg)) {
      const int b = t & 1;
      if (!mbar_wait_warp(accf0 + 8 * b, (uint32_t)(t >> 1) & 1, p.status)) break;
      fence_after();
      const int slab = sg.tile % p.slabs, group = sg.tile / p.slabs;
      const int row0 = group * 256 + (int)rank * 128 + q * 32;  // this warp's 32 rows
      const int o0 = slab * kPairN;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * kPairN);
      float* out = p.part + (size_t)sg.plane * p.rows * p.outs;
      // lane = row: each lane stores its row's 32 columns per chunk as eight 16-byte
      // stores straight from the TMEM registers (a shared-memory transpose into full
      // 128-byte rows was latency-bound)
      const int r = row0 + lane;
      for (int c = c_lo; c < c_lo + ncol; c += 32) {
        uint32_t v0[16], v1[16];
        tmem_ld16_nowait(tbase + c, v0);
        tmem_ld16_nowait(tbase + c + 16, v1);
        tmem_wait_ld();
        if (r < p.rows) {
          float* orow = out + (size_t)r * p.outs + o0 + c;
          auto v = [&](int k) { return __uint_as_float(k < 16 ? v0[k] : v1[k - 16]); };
          if (o0 + c + 32 <= p.outs) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              reinterpret_cast<float4*>(orow)[k] = make_float4(v(4 * k), v(4 * k + 1), v(4 * k + 2), v(4 * k + 3));
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (o0 + c + k < p.outs) orow[k] = v(k);
          }
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(acce_leader + 8 * b)
                     : "memory");
      ++t;
    }
  }
  fence_before();
  __syncthreads();
  cluster_sync_all();  // no copy, commit, arrival or MMA of the pair is outstanding past this point
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kPairN)
                 : "memory");
  }
}

// ---------------------------------------------------------------- host side

Splits pair_splits(const PairPlan& pl) {
  Splits sp;
  sp.S = pl.S;
  sp.N = kPairN;
  sp.slabs = pl.slabs;
  sp.kb = pl.kblocks;
  sp.G = pl.G;
  sp.U = pl.U;
  return sp;
}

bool use_pair_engine(int rows, int xplanes, int wplanes) {
  // Up to 512 rows (4 TMEM-resident 128-row tiles) the one-CTA engine with
  // uniform split-K measured as fast or faster on the drafter's products
  // (fewer partial planes for the consumers, a cheaper launch); beyond that it
  // has to split the rows into groups that each stream the weights again.
  return xplanes == 1 && wplanes == 1 && rows > 512;
}

PairPlan pair_plan(int rows, int outs, int K, int num_sms) {
  PairPlan best;
  if (rows <= 128 || rows > 4096 || K % 64 || K < 64 || outs % 8 || outs <= 64 || num_sms < 2) return best;
  const int kblocks = K / 64;
  const int slabs = (outs + kPairN - 1) / kPairN;
  const int groups = (rows + 255) / 256;
  const long long tiles = (long long)groups * slabs;
  const long long U = tiles * kblocks;
  const long long pairs = num_sms / 2;
  const int stages0 = (int)((kSmemBudget - 2048 - kPairStaging) / kPairStage);
  // Cost model (seconds): a k block costs ~700 cycles of 2-SM MMA per SM; the
  // weights stream at ~6.5 TB/s per row group; each partial plane is written
  // and read back once; an epilogue drains 128 x 256 floats per CTA.
  const double clk = 1.9e9, hbm = 6.5e12, t_kb = 700.0 / clk, t_epi = 1.5e-6, launch = 3.0e-6;
  const double t_hbm = (double)outs * K * 2.0 * groups / hbm;
  double best_t = 1e30;
  // candidates: G = tiles * S workers (S dividing the k blocks: exactly S planes
  // per tile, several waves if G > pairs), or stream-K with G = pairs
  for (int cand = 0; cand <= 16; ++cand) {
    long long G;
    if (cand == 0) {
      G = U < pairs ? U : pairs;
    } else {
      const int S = cand;
      if (kblocks % S) continue;
      G = tiles * S;
    }
    PairPlan pl;
    pl.kblocks = kblocks;
    pl.slabs = slabs;
    pl.groups = groups;
    pl.U = U;
    pl.G = (int)G;
    pl.stages = stages0 > 8 ? 8 : stages0;
    const Splits sp = pair_splits(pl);
    int smax = 1;
    double mean = 0.0;
    for (long long t = 0; t < tiles; ++t) {
      const long long u0 = t * kblocks;
      const int n = (int)(splits_owner(sp, u0 + kblocks - 1) - splits_owner(sp, u0) + 1);
      smax = n > smax ? n : smax;
      mean += n;
    }
    mean /= (double)tiles;
    pl.S = smax;
    if (smax > 16) continue;
    const long long waves = (G + pairs - 1) / pairs;
    const double per_pair = (double)((U + G - 1) / G) * t_kb + t_epi * (double)((U + G - 1) / G / kblocks + 1);
    double t = (double)waves * per_pair;
    t = (t > t_hbm ? t : t_hbm) + launch + mean * rows * (double)outs * 8.0 / hbm;
    if (t < best_t * 0.999) {
      best_t = t;
      best = pl;
      best.ok = true;
    }
  }
  return best;
}

size_t pair_smem_bytes(const PairPlan& pl) {
  return 1024 /* align */ + 1024 /* barriers */ + (size_t)pl.stages * kPairStage + kPairStaging;
}

cudaError_t launch_pair(const PairPlan& pl, const CUtensorMap* x, const CUtensorMap* w, PairParams prm,
                        cudaStream_t s) {
  if (!pl.ok) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBudget);
  if (e != cudaSuccess) return e;
  prm.kblocks = pl.kblocks;
  prm.slabs = pl.slabs;
  prm.stages = pl.stages;
  prm.U = pl.U;
  prm.G = pl.G;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pl.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pair_smem_bytes(pl);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, tc_pair_kernel, *x, *w, prm);
}

}  // namespace tc
}  // namespace dlite
