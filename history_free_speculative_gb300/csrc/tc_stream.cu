// Persistent stream-K tensor-core GEMM for products with few activation rows
// (<= 128, one bf16 plane each side):
//
//   part[z][r][o]: the product X[r, :] . W[o, :] is the sum over the planes z
//   that the split descriptor (Splits, internal.h) gives for (r, o).
//
// With few rows the product is a stream of the weights; what limits it is how
// evenly and continuously every SM pulls its share. The work is U = slabs x
// k blocks units (N output features x 64-wide k block each) in slab-major
// order and CTA c (one per SM) takes the contiguous units [c U / G, (c+1) U / G):
// every SM streams the same number of weight bytes, in long runs. Each piece of
// a slab (segment) accumulates in one of two TMEM buffers (M = 128, N columns);
// its epilogue writes the rows x N fp32 partial to plane (c - first CTA of the
// slab) while the MMAs of the next segment run in the other buffer. The
// partials are small (rows <= 128), so the extra planes cost little.
//
// Warp roles: warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, warps 2-9
// epilogue (warp w reads TMEM lane quadrant w % 4). Every wait is bounded
// (~2 s of %globaltimer); on expiry the status word is flagged and the roles
// run to the end instead of hanging.
#include "tc_device.cuh"
#include "tc_gemm.h"

namespace dlite {
namespace tc {

constexpr uint32_t kStreamOverhang = 128u * 128u;  // the 128-row MMA operand read from the last stage

struct StreamSeg {
  int slab, kb_lo, n, plane;
};
__device__ __forceinline__ bool stream_next(const StreamParams& p, long long& u, long long end, int cta,
                                            StreamSeg& sg) {
  if (u >= end) return false;
  const long long slab = u / p.kblocks;
  sg.slab = (int)slab;
  sg.kb_lo = (int)(u - slab * p.kblocks);
  const long long lim = (slab + 1) * p.kblocks < end ? (slab + 1) * p.kblocks : end;
  sg.n = (int)(lim - u);
  sg.plane = cta - (int)(((slab * p.kblocks + 1) * p.G - 1) / p.U);  // owner of the slab's first unit
  u = lim;
  return true;
}

template <int N>
__global__ void __launch_bounds__(kThreads, 1)
    tc_stream_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw,
                     const StreamParams p) {
  constexpr uint32_t kWTile = (uint32_t)N * 128u;
  // Shared memory: [barriers | pad to 1 KB] [stage 0] ... [stage S-1] [epilogue staging]
  // stage = [X tile: x_box rows in a_slot_bytes(x_box)][W: N rows x 128 B]
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)base;
  const uint32_t full0 = su32(bars), empty0 = su32(bars + p.stages);
  const uint32_t accf0 = su32(bars + 2 * p.stages), acce0 = su32(bars + 2 * p.stages + 2);
  const uint32_t done = su32(bars + 2 * p.stages + 4);
  uint32_t* tmem_holder = (uint32_t*)(bars + 2 * p.stages + 5);
  uint8_t* smem = base + 1024;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool aborted = p.status && (*(volatile int*)p.status & kDevTimeout);
  const int cta = (int)blockIdx.x;
  const long long u_begin = aborted ? 0 : (long long)cta * p.U / p.G;
  const long long u_end = aborted ? 0 : (long long)(cta + 1) * p.U / p.G;
  const uint32_t a_slot = a_slot_bytes(p.x_box);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 4 * kEpiGroups);
    }
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_holder)),
                 "r"(2 * N)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_trigger();

  if (warp == 0) {  // ---------------- TMA producer
    const uint32_t bytes = kWTile + (uint32_t)p.x_box * 128u;
    auto load = [&](const StreamSeg& sg, int j, int i, bool weights, bool acts) {
      const int s = i % p.stages;
      const uint32_t st = su32(smem + (size_t)s * p.stage_bytes);
      const int kb = sg.kb_lo + j;
      if (weights) {
        mbar_expect_tx(full0 + 8 * s, bytes);
        tma_load_4d(st + a_slot, &mw, full0 + 8 * s, kb, (sg.slab * N) >> 6);
      }
      if (acts) tma_load_2d(st, &mx, full0 + 8 * s, kb * 64, 0);
    };
    // weights do not depend on the previous kernel: request the first stages'
    // weight tiles before waiting for it, then their activation tiles
    {
      long long u = u_begin;
      StreamSeg sg;
      int i = 0;
      while (i < p.stages && stream_next(p, u, u_end, cta, sg))
        for (int j = 0; j < sg.n && i < p.stages; ++j, ++i)
          if (lane == 0) load(sg, j, i, true, false);
      __syncwarp();
      pdl_wait();
      u = u_begin;
      i = 0;
      while (i < p.stages && stream_next(p, u, u_end, cta, sg))
        for (int j = 0; j < sg.n && i < p.stages; ++j, ++i)
          if (lane == 0) load(sg, j, i, false, true);
      __syncwarp();
    }
    long long u = u_begin;
    StreamSeg sg;
    int i = 0;
    bool ok = true;
    int issued = 0;
    while (ok && stream_next(p, u, u_end, cta, sg)) {
      for (int j = 0; j < sg.n; ++j, ++i) {
        if (i < p.stages) {  // issued above
          issued = i + 1;
          continue;
        }
        const int s = i % p.stages;
        if (!mbar_wait_warp(empty0 + 8 * s, (uint32_t)(i / p.stages - 1) & 1, p.status)) {
          ok = false;
          break;
        }
        if (lane == 0) load(sg, j, i, true, true);
        __syncwarp();
        issued = i + 1;
      }
    }
    if (!ok) {  // let the copies still in flight land before the CTA exits
      for (int k = issued - p.stages < 0 ? 0 : issued - p.stages; k < issued; ++k)
        mbar_wait_warp(full0 + 8 * (k % p.stages), (uint32_t)(k / p.stages) & 1, nullptr);
    }
  } else if (warp == 1) {  // ---------------- MMA issuer
    const uint32_t idesc = idesc_bf16(128, N);
    const uint64_t desc0 = sw128_desc(su32(smem));
    const uint64_t sdelta = (uint64_t)(p.stage_bytes >> 4);
    const uint64_t wofs = (uint64_t)(a_slot >> 4);
    long long u = u_begin;
    StreamSeg sg;
    int i = 0, t = 0;
    bool ok = true;
    while (ok && stream_next(p, u, u_end, cta, sg)) {
      const int b = t & 1;
      if (t >= 2 && !mbar_wait_warp(acce0 + 8 * b, (uint32_t)((t >> 1) - 1) & 1, p.status)) break;
      fence_after();
      const uint32_t dcol = tmem + (uint32_t)(b * N);
      for (int j = 0; j < sg.n; ++j, ++i) {
        const int s = i % p.stages;
        if (!mbar_wait_warp(full0 + 8 * s, (uint32_t)(i / p.stages) & 1, p.status)) {
          ok = false;
          break;
        }
        fence_after();
        if (lane == 0) {
          const uint64_t a0 = desc0 + sdelta * (uint64_t)s;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // +32 B along K = +2 in the encoded start address
            umma_bf16(dcol, a0 + (uint64_t)(kk * 2), a0 + wofs + (uint64_t)(kk * 2), idesc,
                      (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(empty0 + 8 * s);
        }
        __syncwarp();
      }
      // also after an expired wait, so that the epilogue runs to the end
      if (lane == 0) umma_commit(accf0 + 8 * b);
      __syncwarp();
      ++t;
    }
    // every product issued has finished before TMEM is released
    if (lane == 0) umma_commit(done);
    __syncwarp();
    mbar_wait_warp(done, 0, nullptr);
  } else {  // ---------------- epilogue warps 2 .. 9
    const int q = warp & 3;
    const int eg = (warp - 2) >> 2;
    const int ncol = N / kEpiGroups;
    const int c_lo = eg * ncol;
    const int row0 = q * 32;  // this warp's 32 rows
    const int row = row0 + lane;
    const bool live = row < p.rows;
    pdl_wait();  // the partial buffer may still be read by the previous kernel
    long long u = u_begin;
    StreamSeg sg;
    int t = 0;
    while (stream_next(p, u, u_end, cta, sg)) {
      const int b = t & 1;
      if (!mbar_wait_warp(accf0 + 8 * b, (uint32_t)(t >> 1) & 1, p.status)) break;
      fence_after();
      if (row0 < p.rows) {  // a warp whose rows are all past the end only keeps the protocol
        const int o0 = sg.slab * N;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * N);
        // lane = row: each live lane stores its row's 32 columns per chunk as
        // eight 16-byte stores straight from the TMEM registers (few rows: a
        // handful of instructions per warp instead of a shared-memory transpose)
        float* orow = p.part + ((size_t)sg.plane * p.rows + (live ? row : 0)) * p.outs + o0;
        for (int c = c_lo; c < c_lo + ncol; c += 32) {
          uint32_t v0[16], v1[16];
          tmem_ld16_nowait(tbase + c, v0);
          tmem_ld16_nowait(tbase + c + 16, v1);
          tmem_wait_ld();
          auto v = [&](int k) { return __uint_as_float(k < 16 ? v0[k] : v1[k - 16]); };
          if (live) {
            if (o0 + c + 32 <= p.outs) {
              float4* dst = reinterpret_cast<float4*>(orow + c);
#pragma unroll
              for (int k = 0; k < 8; ++k)
                dst[k] = make_float4(v(4 * k), v(4 * k + 1), v(4 * k + 2), v(4 * k + 3));
            } else {
#pragma unroll
              for (int k = 0; k < 32; ++k)
                if (o0 + c + k < p.outs) orow[c + k] = v(k);
            }
          }
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce0 + 8 * b);
      ++t;
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * N) : "memory");
  }
}

// ---------------------------------------------------------------- host side

bool use_stream_engine(int rows, int xplanes, int wplanes) {
  return xplanes == 1 && wplanes == 1 && rows >= 1 && rows <= 128;
}

Splits stream_splits(const StreamPlan& pl) {
  Splits sp;
  sp.S = pl.S;
  sp.N = pl.N;
  sp.slabs = pl.slabs;
  sp.kb = pl.kblocks;
  sp.G = pl.G;
  sp.U = pl.U;
  return sp;
}

StreamPlan stream_plan(int rows, int outs, int K, int num_sms) {
  StreamPlan pl;
  if (rows < 1 || rows > 128 || K % 64 || K < 64 || outs % 8 || num_sms < 1) return pl;
  const int wrows = (outs + 63) / 64 * 64;  // tiled weight rows
  pl.N = 256;
  while (pl.N > 64 && pl.N > wrows) pl.N >>= 1;
  pl.x_box = (rows + 7) / 8 * 8;
  pl.kblocks = K / 64;
  pl.slabs = (outs + pl.N - 1) / pl.N;
  pl.U = (long long)pl.slabs * pl.kblocks;
  pl.G = (int)(pl.U < num_sms ? pl.U : num_sms);
  pl.stage_bytes = (uint32_t)pl.N * 128u + a_slot_bytes(pl.x_box);
  // the 128-row MMA operand of the x_box-row activation tile overhangs into the
  // weight tile behind it (stale bytes feeding unused TMEM lanes); behind the
  // last stage a pad takes the overhang
  pl.tail_pad = kStreamOverhang;
  int stages = (int)((kSmemBudget - 2048 - pl.tail_pad) / pl.stage_bytes);
  if (stages > 8) stages = 8;
  if (stages < 2) return pl;
  pl.stages = stages;
  const Splits sp = stream_splits(pl);
  int smax = 1;
  for (long long s = 0; s < pl.slabs; ++s) {
    const long long u0 = s * pl.kblocks;
    const int n = (int)(splits_owner(sp, u0 + pl.kblocks - 1) - splits_owner(sp, u0) + 1);
    smax = n > smax ? n : smax;
  }
  pl.S = smax;
  pl.ok = smax <= 16;
  return pl;
}

size_t stream_smem_bytes(const StreamPlan& pl) {
  return 1024 /* align */ + 1024 /* barriers */ + (size_t)pl.stages * pl.stage_bytes + pl.tail_pad;
}

cudaError_t launch_stream(const StreamPlan& pl, const CUtensorMap* x, const CUtensorMap* w, StreamParams prm,
                          cudaStream_t s) {
  if (!pl.ok) return cudaErrorInvalidValue;
  void (*fn)(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap, const StreamParams) =
      pl.N == 256 ? tc_stream_kernel<256> : pl.N == 128 ? tc_stream_kernel<128> : tc_stream_kernel<64>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
  if (e != cudaSuccess) return e;
  prm.kblocks = pl.kblocks;
  prm.stages = pl.stages;
  prm.stage_bytes = pl.stage_bytes;
  prm.x_box = pl.x_box;
  prm.U = pl.U;
  prm.G = pl.G;
  return launch_pdl(fn, dim3(pl.G), dim3(kThreads), stream_smem_bytes(pl), s, *x, *w, prm);
}

}  // namespace tc
}  // namespace dlite
