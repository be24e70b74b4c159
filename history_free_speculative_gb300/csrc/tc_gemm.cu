// Tensor-core GEMM engine for sm_103a: TMA -> shared memory (128B swizzle)
// -> tcgen05.mma (bf16 x bf16 -> fp32 in TMEM) -> tcgen05.ld epilogue.
//
//   D[r, o] = sum_k X[r, k] * W[o, k]
// X (activations, A operand): rows in M-tiles of 128 (TMEM lanes).
// W (weights, B operand): one slab of N output features per CTA (TMEM columns).
// Every CTA streams its weight slab exactly once; all M-tiles of its row
// group are accumulated side by side in TMEM, so weights are never re-read.
// Warp roles: warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer (one
// thread), warps 2-5 = epilogue (warp w reads TMEM lanes 32*(w%4)..+31).
// Every mbarrier wait is bounded (~2 s of %globaltimer); on expiry the kernel
// flags the device status word and runs to its end instead of hanging.
#include "tc_device.cuh"

#include "tc_gemm.h"

namespace dlite {
namespace tc {

// NMT: M-tiles per CTA; XP / WP: bf16 planes of X / W (products x0w0, + x1w0, + x0w1).
// The MMA issue loop is fully unrolled over these so the issuing thread only
// adds precomputed descriptor offsets between tcgen05.mma instructions.
template <int NMT, int XP, int WP>
__global__ void __launch_bounds__(kGemmThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap mx0, const __grid_constant__ CUtensorMap mx1,
                   const __grid_constant__ CUtensorMap mw0, const __grid_constant__ CUtensorMap mw1,
                   const __grid_constant__ CUtensorMap mo, const TcParams p) {
  // Shared memory: [barriers | pad to 1 KB] [stage 0] ... [stage S-1] [tail pad].
  // Stage: [activation slots: NMT x XP x a_slot] [weight planes: WP x N rows x 128 B].
  // An activation slot holds only the x_box loaded rows; with fewer than 128 the
  // 128-row MMA operand overhangs into the following bytes (stale data feeding
  // only unused TMEM lanes), and the tail pad keeps that overhang inside the
  // allocation (full 128-row slots need none: one more stage fits).
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)base;
  uint32_t* tmem_holder = (uint32_t*)(bars + 2 * p.stages + 1);
  uint8_t* smem = base + 1024;
  const uint32_t full0 = su32(bars), empty0 = su32(bars + p.stages), accf = su32(bars + 2 * p.stages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int o0 = blockIdx.x * p.N;
  const int split = blockIdx.y;
  const int m0 = blockIdx.z * p.n_mt * 128;
  if (p.skip_row0 > 0 && m0 >= p.skip_row0 && o0 + p.N <= p.skip_cols) {  // a tile nobody reads
    pdl_trigger();
    return;
  }
  // After any bounded wait has expired on this device, later CTAs skip their
  // work (and only allocate / free TMEM) so a broken launch ends quickly.
  const bool aborted = p.status && (*(volatile int*)p.status & kDevTimeout);
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(kb0 + p.kb_per_split, p.kblocks);
  const int nkb = aborted ? 0 : kb1 - kb0;
  const int rot = nkb > 0 ? (int)(blockIdx.x % (unsigned)nkb) : 0;
  const uint32_t wtile = (uint32_t)p.N * 128u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accf, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_holder)),
                 "r"(p.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_trigger();

  // Role loops run with the whole warp converged: every lane waits on the
  // barrier, one lane issues (a lone active lane beside 31 lanes parked at a
  // block barrier issues far more slowly).
  if (warp == 0) {  // ---------------- TMA producer
    // activation tiles are p.x_box rows tall (only the valid rows when rows < 128; the
    // rest of the 128-row smem tile holds stale data that only feeds unused TMEM lanes)
    const uint32_t bytes = (uint32_t)WP * wtile + (uint32_t)(NMT * XP) * (uint32_t)p.x_box * 128u;
    const uint32_t a_slot = a_slot_bytes(p.x_box);
    // k blocks in a per-CTA rotated order: concurrent CTAs fetch different
    // activation tiles instead of all hitting the same L2 lines
    // One lane issues every copy, so its per-stage instruction latency bounds
    // the stream: stage, phase and k block advance by increments (integer
    // division by a runtime divisor costs tens of cycles). kr = (i + rot) % nkb.
    auto load_w = [&](int kr, int s) {
      const uint32_t st = su32(smem + (size_t)s * p.stage_bytes);
      const uint32_t fb = full0 + 8 * s;
      const int kb = kb0 + kr;
      mbar_expect_tx(fb, bytes);
      const uint32_t wst = st + (uint32_t)(NMT * XP) * a_slot;
      tma_load_4d(wst, &mw0, fb, kb, o0 >> 6);
      if (WP == 2) tma_load_4d(wst + wtile, &mw1, fb, kb, o0 >> 6);
    };
    auto load_x = [&](int kr, int s) {
      const uint32_t st = su32(smem + (size_t)s * p.stage_bytes);
      const uint32_t fb = full0 + 8 * s;
      const int kx = (kb0 + kr) * 64;
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
        for (int pl = 0; pl < XP; ++pl)
          tma_load_2d(st + (uint32_t)(mt * XP + pl) * a_slot, pl ? &mx1 : &mx0, fb, kx, m0 + mt * 128);
    };
    // Weights do not depend on the previous kernel: stream the first stages'
    // weight tiles before waiting for it, then the activations.
    const int pre = nkb < p.stages ? nkb : p.stages;
    if (lane == 0)
      for (int i = 0, kr = rot; i < pre; ++i) {
        load_w(kr, i);
        if (++kr == nkb) kr = 0;
      }
    __syncwarp();
    pdl_wait();
    if (lane == 0)
      for (int i = 0, kr = rot; i < pre; ++i) {
        load_x(kr, i);
        if (++kr == nkb) kr = 0;
      }
    __syncwarp();
    // cursor of copy i = pre: stage s, the phase ph of its use, k block kr
    int s = pre == p.stages ? 0 : pre, kr = pre + rot >= nkb ? pre + rot - nkb : pre + rot;
    uint32_t ph = pre == p.stages ? 1u : 0u;
    for (int i = pre; i < nkb; ++i) {
      // the slot's previous use (copy i - stages) had the other phase
      if (!mbar_wait_warp(empty0 + 8 * s, ph ^ 1u, p.status)) break;
      if (lane == 0) {
        load_w(kr, s);
        load_x(kr, s);
      }
      __syncwarp();
      if (++s == p.stages) {
        s = 0;
        ph ^= 1u;
      }
      if (++kr == nkb) kr = 0;
    }
  } else if (warp == 1) {  // ---------------- MMA issuer
    constexpr int kCombos = 1 + (XP == 2) + (WP == 2);
    const uint32_t idesc = idesc_bf16(128, p.N);
    uint32_t dcol[NMT];
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt) dcol[mt] = tmem + (uint32_t)(mt * p.N);
    const uint32_t a_slot = a_slot_bytes(p.x_box);
    const uint64_t wdelta = (uint64_t)(wtile >> 4);                      // second weight plane
    const uint64_t wbase = (uint64_t)(((uint32_t)(NMT * XP) * a_slot) >> 4);  // weights follow the activations
    const uint64_t aslot = (uint64_t)(a_slot >> 4);
    const uint64_t desc0 = sw128_desc(su32(smem));
    const uint64_t sdelta = (uint64_t)(p.stage_bytes >> 4);
    int s = 0;  // stage of k block i and the phase of its use
    uint32_t ph = 0;
    for (int i = 0; i < nkb; ++i) {
      if (!mbar_wait_warp(full0 + 8 * s, ph, p.status)) break;
      fence_after();
      if (lane == 0) {
        const uint64_t a0 = desc0 + sdelta * (uint64_t)s;
        const uint64_t b0 = a0 + wbase;
        const uint32_t first = i > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
          for (int mt = 0; mt < NMT; ++mt) {
#pragma unroll
            for (int c = 0; c < kCombos; ++c) {
              const int px = (XP == 2 && c == 1) ? 1 : 0;
              const int pw = (WP == 2 && c == kCombos - 1 && c > 0) ? 1 : 0;
              // +32 B along K inside the 128-byte swizzled row = +2 in the encoded start address
              const uint64_t ad = a0 + (uint64_t)(kk * 2) + (uint64_t)(mt * XP + px) * aslot;
              const uint64_t bd = b0 + (uint64_t)(kk * 2) + (pw ? wdelta : 0ull);
              umma_bf16(dcol[mt], ad, bd, idesc, (kk > 0 || c > 0) ? 1u : first);
            }
          }
        }
        umma_commit(empty0 + 8 * s);
      }
      __syncwarp();
      if (++s == p.stages) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (lane == 0) umma_commit(accf);
    __syncwarp();
  } else {  // ---------------- epilogue warps 2 .. 2 + 4 * kGemmEpiGroups - 1
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int eg = (warp - 2) >> 2;                 // column group of this warp
    const int ncol = p.N / kGemmEpiGroups;          // columns per group (multiple of 16)
    const int c_lo = eg * ncol, c_hi = c_lo + ncol;
    const bool got = mbar_wait_warp(accf, 0, p.status);
    fence_after();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // stage memory is reused below
    pdl_wait();  // outputs may still be read by the previous kernel
    if (got) {
      for (int mt = 0; mt < NMT; ++mt) {
        const int r = m0 + mt * 128 + q * 32 + lane;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(mt * p.N);
        if (p.mode == 0 && p.tma_out && ncol % 32 == 0) {
          // lane = row of a 32 x 32 box staged in this warp's 4 KB of the idle
          // stage memory (128-byte swizzle: 16-byte chunk j of row L at chunk
          // j ^ (L & 7), so the lanes' stores spread over the banks), written
          // by one bulk tensor store; rows past p.rows are clipped by the map
          const uint32_t stg = su32(smem + (size_t)(warp - 2) * 4096);
          const int row0 = m0 + mt * 128 + q * 32;
          for (int c = c_lo; c < c_hi; c += 32) {
            uint32_t v0[16], v1[16];
            tmem_ld16_nowait(tbase + c, v0);
            tmem_ld16_nowait(tbase + c + 16, v1);
            tmem_wait_ld();
            if (lane == 0) bulk_wait_read0();  // the previous box has left the buffer
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t a = stg + (uint32_t)lane * 128u + (uint32_t)((j ^ (lane & 7)) * 16);
              const uint32_t w0 = j < 4 ? v0[4 * j] : v1[4 * (j - 4)];
              const uint32_t w1 = j < 4 ? v0[4 * j + 1] : v1[4 * (j - 4) + 1];
              const uint32_t w2 = j < 4 ? v0[4 * j + 2] : v1[4 * (j - 4) + 2];
              const uint32_t w3 = j < 4 ? v0[4 * j + 3] : v1[4 * (j - 4) + 3];
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w0), "r"(w1), "r"(w2),
                           "r"(w3)
                           : "memory");
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0 && row0 < p.rows && o0 + c < p.outs) {
              tma_store_3d(&mo, stg, o0 + c, row0, split);
              bulk_commit();
            }
          }
          if (lane == 0) bulk_wait0();  // performed before the CTA ends
          __syncwarp();
        } else if (p.mode == 0) {
          // lane = row: each lane stores its row's 16 columns per chunk as four
          // 16-byte stores straight from the TMEM registers (measured faster than
          // a shared-memory transpose into full 128-byte rows: the epilogue is
          // bound by its instruction latency, not by the store pattern)
          float* out = p.part + (size_t)split * p.rows * p.outs;
          for (int c = c_lo; c < c_hi; c += 16) {
            uint32_t v0[16];
            tmem_ld16_nowait(tbase + c, v0);
            tmem_wait_ld();
            if (r < p.rows) {
              float* orow = out + (size_t)r * p.outs + o0 + c;
              if (o0 + c + 16 <= p.outs) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  reinterpret_cast<float4*>(orow)[k] =
                      make_float4(__uint_as_float(v0[4 * k]), __uint_as_float(v0[4 * k + 1]),
                                  __uint_as_float(v0[4 * k + 2]), __uint_as_float(v0[4 * k + 3]));
              } else {
#pragma unroll
                for (int k = 0; k < 16; ++k)
                  if (o0 + c + k < p.outs) orow[k] = __uint_as_float(v0[k]);
              }
            }
          }
        } else if (p.mode == 3) {
          // residual: lane = row stores res + product of its row's 16 columns per
          // chunk as fp32 (and the tap) and as the hi / lo bf16 planes
          for (int c = c_lo; c < c_hi; c += 16) {
            uint32_t v0[16];
            tmem_ld16_nowait(tbase + c, v0);
            tmem_wait_ld();
            if (r < p.rows && o0 + c < p.outs) {
              const size_t idx = (size_t)r * p.outs + o0 + c;  // outs is a multiple of 16 here
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float4 b4 = *reinterpret_cast<const float4*>(p.res + idx + 4 * k);
                const float4 v = make_float4(b4.x + __uint_as_float(v0[4 * k]), b4.y + __uint_as_float(v0[4 * k + 1]),
                                             b4.z + __uint_as_float(v0[4 * k + 2]),
                                             b4.w + __uint_as_float(v0[4 * k + 3]));
                *reinterpret_cast<float4*>(p.out32 + idx + 4 * k) = v;
                if (p.tap32) *reinterpret_cast<float4*>(p.tap32 + idx + 4 * k) = v;
                bf16 h[4], l[4];
                split_bf16(v.x, h[0], l[0]);
                split_bf16(v.y, h[1], l[1]);
                split_bf16(v.z, h[2], l[2]);
                split_bf16(v.w, h[3], l[3]);
                *reinterpret_cast<uint2*>(p.act[0] + idx + 4 * k) = *reinterpret_cast<const uint2*>(h);
                *reinterpret_cast<uint2*>(p.act[1] + idx + 4 * k) = *reinterpret_cast<const uint2*>(l);
              }
            }
          }
        } else if (p.mode == 2) {
          // SwiGLU: the slab's columns come in blocks of 64, [32 gate | 32 up] of the
          // same 32 features; lane = row stores a = silu(gate) * up of its row's 32
          // features as bf16 (16-byte stores straight from the registers)
          const int F = p.outs / 2;
          for (int blk = eg; blk < p.N / 64; blk += kGemmEpiGroups) {
            uint32_t g0[16], g1[16], u0[16], u1[16];
            tmem_ld16_nowait(tbase + blk * 64, g0);
            tmem_ld16_nowait(tbase + blk * 64 + 16, g1);
            tmem_ld16_nowait(tbase + blk * 64 + 32, u0);
            tmem_ld16_nowait(tbase + blk * 64 + 48, u1);
            tmem_wait_ld();
            const int f0 = (o0 / 64 + blk) * 32;  // the block's first feature (F is a multiple of 32)
            if (r < p.rows && f0 < F) {
              const size_t idx = (size_t)r * F + f0;
#pragma unroll
              for (int k = 0; k < 4; ++k) {  // 8 features per 16-byte store
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  float a2[2];
#pragma unroll
                  for (int t2 = 0; t2 < 2; ++t2) {
                    const int j = 8 * k + 2 * e + t2;
                    const float g = __uint_as_float(j < 16 ? g0[j] : g1[j - 16]);
                    const float u = __uint_as_float(j < 16 ? u0[j] : u1[j - 16]);
                    // fast exponential and division (a few ulp of fp32, far below the
                    // bf16 rounding of the stored activation): this epilogue runs after
                    // the last product of the tile, unhidden; silu -> -0 when exp overflows
                    a2[t2] = __fdividef(g, 1.f + __expf(-g)) * u;
                  }
                  bf16 h0, l0, h1, l1;
                  if (p.act_planes == 2) {
                    split_bf16(a2[0], h0, l0);
                    split_bf16(a2[1], h1, l1);
                  } else {
                    h0 = __float2bfloat16_rn(a2[0]);
                    h1 = __float2bfloat16_rn(a2[1]);
                    l0 = l1 = h0;
                  }
                  hw[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                  lw[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
                }
                reinterpret_cast<uint4*>(p.act[0] + idx)[k] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                if (p.act_planes == 2)
                  reinterpret_cast<uint4*>(p.act[1] + idx)[k] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
              }
            }
          }
        } else {
          // LM head: 4 best (score, id) and LSE partials of this vocabulary slab for row r
          const bool sampling = p.inv_T > 0.f;
          const float c2s = p.inv_T * kLog2e;
          LmAcc acc;
          lm_acc_init(acc);
          const bool valid = r < p.rows;
          PhiloxRow pr = {0u, 0u, 0u};
          if (sampling && valid) {
            const int req = r / p.K_draft;
            const uint32_t pos = (uint32_t)(p.pos[req] + (r % p.K_draft) + 1);
            pr = philox_row_init(pos, (uint32_t)req, kTagGumbel, p.k0, p.k1);
          }
          for (int c = c_lo; c < c_hi; c += 16) {
            uint32_t raw[16];
            tmem_ld16_nowait(tbase + c, raw);  // warp-collective: executed by every lane
            tmem_wait_ld();
            const int v0 = o0 + c;
            const int nv = p.outs - v0;  // outs is a multiple of 8: whole groups of 4 only
            if (nv > 0) {                 // uniform across the warp; rows differ per lane
              if (nv >= 16) {
                if (sampling)
                  lm_fold16<true, true>(acc, raw, v0, 16, c2s, pr, p.k0, p.k1, valid);
                else
                  lm_fold16<false, true>(acc, raw, v0, 16, c2s, pr, p.k0, p.k1, valid);
              } else {
                if (sampling)
                  lm_fold16<true, false>(acc, raw, v0, nv, c2s, pr, p.k0, p.k1, valid);
                else
                  lm_fold16<false, false>(acc, raw, v0, nv, c2s, pr, p.k0, p.k1, valid);
              }
            }
          }
          if (valid) lm_acc_store(acc, p.rec + ((size_t)blockIdx.x * kGemmEpiGroups + eg) * p.rows + r);
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tmem_cols)
                 : "memory");
  }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

static EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)f;
  }
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows) {
  EncodeTiledFn fn = encoder();
  if (!fn || !base || ((uintptr_t)base & 15) || K % 64 || box_rows < 1 || box_rows > 256 ||
      rows < box_rows)
    return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_out_map(CUtensorMap* m, const void* base, int S, int rows, int outs) {
  EncodeTiledFn fn = encoder();
  if (!fn || !base || ((uintptr_t)base & 15) || S < 1 || rows < 1 || outs < 8 || outs % 4) return false;
  cuuint64_t dims[3] = {(cuuint64_t)outs, (cuuint64_t)rows, (cuuint64_t)S};
  cuuint64_t strides[2] = {(cuuint64_t)outs * 4, (cuuint64_t)rows * outs * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_tiled(CUtensorMap* m, const void* base, int rows, int K, int box_rows) {
  EncodeTiledFn fn = encoder();
  if (!fn || !base || ((uintptr_t)base & 15) || K % 64 || rows % 64 || box_rows % 64 || box_rows < 64 ||
      box_rows > 256 || rows < box_rows)
    return false;
  const int kb = K / 64;
  cuuint64_t dims[4] = {64, 64, (cuuint64_t)kb, (cuuint64_t)(rows / 64)};
  cuuint64_t strides[3] = {128, 8192, (cuuint64_t)kb * 8192};
  cuuint32_t box[4] = {64, 64, 1, (cuuint32_t)(box_rows / 64)};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int next_pow2_cols(int c) {
  int n = 32;
  while (n < c) n <<= 1;
  return n;
}

Plan plan(int rows, int outs, int K, int xplanes, int wplanes, bool lm, bool one_split, int skip_row0,
          int skip_cols) {
  Plan best;
  best.ok = false;
  const int kblocks = K / 64;
  const int mt_total = (rows + 127) / 128;
  const int n_sms = device_sms();
  const double bw_total = 6.5e12, l2_total = 1.6e13, mma_sm = 1.8e15 / n_sms;
  double best_t = 1e30;
  const int combos = 1 + (xplanes == 2) + (wplanes == 2);
  const int nmax_out = ((outs + 63) / 64) * 64;  // tiled weights: rows padded to 64
  for (int gmax = 4; gmax >= 1; gmax >>= 1) {
    const int groups = (mt_total + gmax - 1) / gmax;
    const int n_mt = (mt_total + groups - 1) / groups;
    for (int N = 64; N <= 256; N += 64) {
      if (N * n_mt > 512 || N > nmax_out) continue;  // weight buffers hold >= nmax_out rows
      const uint32_t sb = (uint32_t)wplanes * N * 128 + (uint32_t)n_mt * xplanes * a_slot_bytes(x_box_rows(rows));
      const uint32_t pad = x_box_rows(rows) < 128 ? (uint32_t)kTailPad : 0u;
      int stages = (int)((kSmemBudget - 2048 - pad) / sb);
      if (stages > 8) stages = 8;
      if (stages < 2) continue;
      const int slabs = (outs + N - 1) / N;
      // at most 4 k-splits (every consumer sums the splits on its critical path),
      // up to 16 for few rows, whose partial planes are small: a weight stream
      // then needs the splits to fill the SMs with wide slabs
      const int scap = rows <= 64 ? 16 : 4;
      const int smax = (lm || one_split) ? 1 : (kblocks < scap ? kblocks : scap);
      for (int S = 1; S <= smax; ++S) {
        const int kbps = (kblocks + S - 1) / S;
        const int Se = (kblocks + kbps - 1) / kbps;
        if (Se != S) continue;
        long units = 0;  // CTAs with work (tiles past skip_row0 x before skip_cols are skipped)
        for (int g = 0; g < groups; ++g)
          units += (long)Se * (skip_row0 > 0 && g * n_mt * 128 >= skip_row0 ? slabs - skip_cols / N : slabs);
        const long waves = (units + n_sms - 1) / n_sms;
        const double active = units < n_sms ? (double)units : (double)n_sms;
        double bw_sm = bw_total / active;
        if (bw_sm > 1.2e11) bw_sm = 1.2e11;
        double l2_sm = l2_total / active;  // activation tiles come from L2, shared by all CTAs
        if (l2_sm > 1.5e11) l2_sm = 1.5e11;
        const double t_load = (double)wplanes * N * 128 / bw_sm;
        const double t_l2 = (double)n_mt * xplanes * x_box_rows(rows) * 128 / l2_sm;
        const double t_mma = (double)n_mt * combos * 128.0 * N * 64 * 2 / mma_sm;
        double t_kb = t_load > t_mma ? t_load : t_mma;
        t_kb = (t_kb > t_l2 ? t_kb : t_l2) + 3.0e-8;
        double t = waves * (kbps * t_kb + 2.0e-6);
        if (Se > 1) t += (double)Se * rows * outs * 8.0 / bw_total;
        if (t < best_t * 0.999) {
          best_t = t;
          best.ok = true;
          best.N = N;
          best.S = Se;
          best.kb_per_split = kbps;
          best.kblocks = kblocks;
          best.n_mt = n_mt;
          best.groups = groups;
          best.stages = stages;
          best.stage_bytes = sb;
          best.tail_pad = pad;
          best.tmem_cols = next_pow2_cols(N * n_mt);
        }
      }
    }
  }
  return best;
}

std::vector<Plan> plan_candidates(int rows, int outs, int K, int xplanes, int wplanes, bool one_split) {
  std::vector<Plan> out;
  const int kblocks = K / 64;
  const int mt_total = (rows + 127) / 128;
  const int nmax_out = ((outs + 63) / 64) * 64;
  int prev_nmt = 0;
  for (int gmax = 4; gmax >= 1; gmax >>= 1) {
    const int groups = (mt_total + gmax - 1) / gmax;
    const int n_mt = (mt_total + groups - 1) / groups;
    if (n_mt == prev_nmt) continue;  // the same split of the M-tiles
    prev_nmt = n_mt;
    for (int N = 64; N <= 256; N += 64) {
      if (N * n_mt > 512 || N > nmax_out) continue;
      const uint32_t sb = (uint32_t)wplanes * N * 128 + (uint32_t)n_mt * xplanes * a_slot_bytes(x_box_rows(rows));
      const uint32_t pad = x_box_rows(rows) < 128 ? (uint32_t)kTailPad : 0u;
      int stages = (int)((kSmemBudget - 2048 - pad) / sb);
      if (stages > 8) stages = 8;
      if (stages < 2) continue;
      const int scap = rows <= 64 ? 16 : 4;
      const int smax = one_split ? 1 : (kblocks < scap ? kblocks : scap);
      for (int S = 1; S <= smax; ++S) {
        const int kbps = (kblocks + S - 1) / S;
        if ((kblocks + kbps - 1) / kbps != S) continue;
        Plan p;
        p.ok = true;
        p.N = N;
        p.S = S;
        p.kb_per_split = kbps;
        p.kblocks = kblocks;
        p.n_mt = n_mt;
        p.groups = groups;
        p.stages = stages;
        p.stage_bytes = sb;
        p.tail_pad = pad;
        p.tmem_cols = next_pow2_cols(N * n_mt);
        out.push_back(p);
      }
    }
  }
  return out;
}

size_t smem_bytes(const Plan& pl) {
  // the epilogue reuses the first 64 KB of the stage memory as staging boxes (4 KB per warp)
  size_t stage_mem = (size_t)pl.stages * pl.stage_bytes + pl.tail_pad;
  if (stage_mem < 65536) stage_mem = 65536;
  return 1024 /* align */ + 1024 /* barriers */ + stage_mem;
}

typedef void (*KernelFn)(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap,
                         const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap,
                         const __grid_constant__ CUtensorMap, const TcParams);

template <int NMT>
static KernelFn pick_planes(int xp, int wp) {
  if (xp == 1 && wp == 1) return tc_gemm_kernel<NMT, 1, 1>;
  if (xp == 2 && wp == 1) return tc_gemm_kernel<NMT, 2, 1>;
  if (xp == 2 && wp == 2) return tc_gemm_kernel<NMT, 2, 2>;
  return nullptr;
}

static KernelFn pick(int nmt, int xp, int wp) {
  switch (nmt) {
    case 1: return pick_planes<1>(xp, wp);
    case 2: return pick_planes<2>(xp, wp);
    case 3: return pick_planes<3>(xp, wp);
    case 4: return pick_planes<4>(xp, wp);
    default: return nullptr;
  }
}

cudaError_t launch(const Plan& pl, const CUtensorMap* x0, const CUtensorMap* x1, const CUtensorMap* w0,
                   const CUtensorMap* w1, TcParams prm, cudaStream_t s, const CUtensorMap* out) {
  KernelFn fn = pick(pl.n_mt, prm.xplanes, prm.wplanes);
  if (!fn) return cudaErrorInvalidValue;
  static bool attr[5][3] = {};
  const int pi = prm.xplanes == 1 ? 0 : (prm.wplanes == 1 ? 1 : 2);
  if (!attr[pl.n_mt][pi]) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBudget);
    if (e != cudaSuccess) return e;
    attr[pl.n_mt][pi] = true;
  }
  prm.N = pl.N;
  prm.n_mt = pl.n_mt;
  prm.kb_per_split = pl.kb_per_split;
  prm.kblocks = pl.kblocks;
  prm.stages = pl.stages;
  prm.stage_bytes = pl.stage_bytes;
  prm.tmem_cols = (uint32_t)pl.tmem_cols;
  prm.tma_out = (out && prm.mode == 0) ? 1 : 0;
  dim3 grid((prm.outs + pl.N - 1) / pl.N, pl.S, pl.groups);
  return launch_pdl(fn, grid, dim3(kGemmThreads), smem_bytes(pl), s, *x0, x1 ? *x1 : *x0, *w0,
                    w1 ? *w1 : *w0, out ? *out : *x0, prm);
}

}  // namespace tc
}  // namespace dlite
