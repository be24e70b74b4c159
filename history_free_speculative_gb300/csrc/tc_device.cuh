// Device-side building blocks of the tcgen05 kernels: bounded mbarrier waits,
// TMA tile loads, shared-memory / instruction descriptors, tcgen05.mma issue
// and commit, TMEM loads, and the LM-head score folding shared by the
// one-slab and the persistent LM-head kernels.
#pragma once

#include <cuda.h>

#include "internal.h"

namespace dlite {
namespace tc {

constexpr uint64_t kTimeoutNs = 2000000000ull;

__device__ __forceinline__ uint32_t su32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on phase `parity`; false after limit_ns (status flagged).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* status,
                                          uint64_t limit_ns = kTimeoutNs) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 128; ++i)
      if (mbar_try(bar, parity)) return true;
    if (gtimer() - t0 > limit_ns) {
      flag_status(status, kDevTimeout);
      return false;
    }
  }
}
// Warp-wide bounded wait: every lane polls, lane 0's view decides, so the
// result is uniform across the warp.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, int* status,
                                               uint64_t limit_ns = kTimeoutNs) {
  if (__shfl_sync(0xffffffffu, (int)mbar_try(bar, parity), 0)) return true;
  const uint64_t t0 = gtimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (__shfl_sync(0xffffffffu, (int)mbar_try(bar, parity), 0)) return true;
    const int expired = __shfl_sync(0xffffffffu, (int)(gtimer() - t0 > limit_ns), 0);
    if (expired) {
      if ((threadIdx.x & 31) == 0) flag_status(status, kDevTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// Bulk tensor store of a shared-memory box to global memory (3-D map), tracked
// by this thread's bulk async-group; the box must not start at a negative
// coordinate, and rows / columns past the map's extent are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// 1-D bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16),
// completing on mbarrier `bar` (expect_tx beforehand).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until this thread's bulk stores have finished reading shared memory (the
// buffer may be rewritten) / have been performed completely.
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Weight tile load from the tiled layout: coordinates (0, 0, k block, 64-row slab).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(0), "r"(0), "r"(c2), "r"(c3)
      : "memory");
}

// ---------------------------------------------------------------- CTA pairs (2-SM MMA)
// A cluster of two CTAs on neighbouring SMs runs one M = 256 MMA: each CTA
// holds its 128 rows of A and half of the N columns of B in its own shared
// memory (same offsets in both), rank 0 issues the MMA, and each CTA's TMEM
// receives its 128 rows of D over all N columns. TMA loads of either CTA
// signal rank 0's barrier; rank 0's commits arrive on both CTAs' barriers.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(0), "r"(0), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                               uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
// Arrive on the barrier at this shared-memory offset in both CTAs of the pair
// once every prior 2-SM MMA of this thread has completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          bar),
      "h"((uint16_t)3)
      : "memory");
}

// Shared-memory matrix descriptor: K-major tile, rows of 128 B, 128-byte
// swizzle, 8-row groups 1024 B apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Issue a 16-column TMEM load without waiting; tmem_wait_ld() completes all
// loads issued so far by this thread (lets two loads overlap their latency).
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// ---------------------------------------------------------------- LM-head score folding
// Every epilogue thread owns one row of h and scans its vocabulary columns in
// increasing id order, keeping the 4 best (score, id) it saw and, when
// sampling, the log-sum-exp partials of its columns.
// Greedy: scores are the logits, ids the vocabulary ids.
// Sampling (the two-level draw): each 16-id chunk k is one entry, scored in
// base-2 units as log2(sum_{v in k} 2^(l2_v)) - log2(-log2 u_k), with
// l2 = logit * log2(e) / T and u_k the chunk's uniform (word k & 3 of
// Philox(k >> 2, position, request, TAG_GUMBEL)); that is
// log2(e) (L_k - log(-log u_k)) + log2(ln 2) with L_k the chunk's natural
// log-mass at temperature T, a fixed increasing map of the chunk's Gumbel-max
// score, so the best entries are the finalist chunks. The LSE partials are
// m = max l2 and s = sum 2^(l2 - m).

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// -log2(u) for the uniform u = ((x >> 9) + 1/2) 2^-23 of a 32-bit draw, with a
// small relative error everywhere. The hardware log2 has an absolute error
// near 1, which would swamp -log2(u) when u is within ~1e-4 of 1: exactly the
// draws that give the largest Gumbel noise. There the complement
// w = 1 - u = ((2^23 - 1 - (x >> 9)) + 1/2) 2^-23 (exact) is used with the
// series -ln(1 - w) = w + w^2/2 + w^3/3 + ..., truncated after w^3
// (truncation < w^4/4, relative < 2^-26 for w < 2^-8); elsewhere
// -log2(u) >= 0.0056 and the hardware log2 is used.
__device__ __forceinline__ float neg_log2_u01(uint32_t x) {
  const uint32_t k = x >> 9;
  const float w = fmaf((float)(0x7fffffu - k), 1.1920928955078125e-07f, 5.9604644775390625e-08f);
  const float u = 1.f - w;  // exact: u has at most 24 significant bits
  const float series = w * fmaf(w, fmaf(w, kLog2e / 3.f, kLog2e / 2.f), kLog2e);
  return w < 0.00390625f ? series : -lg2_approx(u);
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}
// Insert (x, v) into a descending top-k list (ties: lower id ranks first):
// replace the last entry, then bubble it up with constant indices only.
__device__ __forceinline__ void cswap(float (&sc)[kTopK], int (&id)[kTopK], int k) {
  if (better(sc[k + 1], id[k + 1], sc[k], id[k])) {
    const float ts = sc[k];
    const int ti = id[k];
    sc[k] = sc[k + 1];
    id[k] = id[k + 1];
    sc[k + 1] = ts;
    id[k + 1] = ti;
  }
}
__device__ __forceinline__ void topk_insert(float (&sc)[kTopK], int (&id)[kTopK], float x, int v) {
  if (!better(x, v, sc[kTopK - 1], id[kTopK - 1])) return;
  sc[kTopK - 1] = x;
  id[kTopK - 1] = v;
#pragma unroll
  for (int k = kTopK - 2; k >= 0; --k) cswap(sc, id, k);
}

struct LmAcc {
  float sc[kTopK];
  int id[kTopK];
  float m, s;
};
__device__ __forceinline__ void lm_acc_init(LmAcc& a) {
#pragma unroll
  for (int j = 0; j < kTopK; ++j) {
    a.sc[j] = -INFINITY;
    a.id[j] = 0x7fffffff;
  }
  a.m = -INFINITY;
  a.s = 0.f;
}
__device__ __forceinline__ void lm_acc_store(const LmAcc& a, LmRec* dst) {
  LmRec rec;
#pragma unroll
  for (int j = 0; j < kTopK; ++j) {
    rec.sc[j] = a.sc[j];
    rec.id[j] = a.id[j];
  }
  rec.m = a.m;
  rec.s = a.s;
  *dst = rec;
}

// Philox4x32-10 with counter words 1..3 (position, request, tag) fixed for a
// row: the first round's outputs that depend on them only are formed once.
struct PhiloxRow {
  uint32_t a0, a1, t;
};
__device__ __forceinline__ PhiloxRow philox_row_init(uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                                     uint32_t k1) {
  const uint64_t p1 = (uint64_t)kPhiloxM1 * c2;
  PhiloxRow r;
  r.a0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
  r.a1 = (uint32_t)p1;
  r.t = c3 ^ k1;
  return r;
}
__device__ __forceinline__ uint4 philox_row(uint32_t c0, const PhiloxRow& pr, uint32_t k0, uint32_t k1) {
  const uint64_t p0 = (uint64_t)kPhiloxM0 * c0;
  uint32_t x0 = pr.a0, x1 = pr.a1, x2 = (uint32_t)(p0 >> 32) ^ pr.t, x3 = (uint32_t)p0;
#pragma unroll
  for (int r = 1; r < 10; ++r) {
    const uint32_t ka = k0 + (uint32_t)r * kPhiloxW0, kb = k1 + (uint32_t)r * kPhiloxW1;
    const uint64_t q0 = (uint64_t)kPhiloxM0 * x0;
    const uint64_t q1 = (uint64_t)kPhiloxM1 * x2;
    const uint32_t n0 = (uint32_t)(q1 >> 32) ^ x1 ^ ka;
    const uint32_t n2 = (uint32_t)(q0 >> 32) ^ x3 ^ kb;
    x1 = (uint32_t)q1;
    x3 = (uint32_t)q0;
    x0 = n0;
    x2 = n2;
  }
  return make_uint4(x0, x1, x2, x3);
}

// Insert (x, v) into the descending list of a thread that scans ids in
// increasing order: every id already held is lower than v, so on equal scores
// the held entry stays first (the lower-id-first order) and only strictly
// greater scores move. Branch-free: the 32 lanes of a warp hold 32 different
// rows, and a branch taken by any one lane would cost the whole warp.
__device__ __forceinline__ void topk_push_scan(LmAcc& a, float x, int v) {
  static_assert(kTopK == 4, "unrolled for 4 entries");
  const bool c0 = x > a.sc[0], c1 = x > a.sc[1], c2 = x > a.sc[2], c3 = x > a.sc[3];
  const float s0 = a.sc[0], s1 = a.sc[1], s2 = a.sc[2];
  const int i0 = a.id[0], i1 = a.id[1], i2 = a.id[2];
  a.sc[3] = c2 ? s2 : (c3 ? x : a.sc[3]);
  a.id[3] = c2 ? i2 : (c3 ? v : a.id[3]);
  a.sc[2] = c1 ? s1 : (c2 ? x : s2);
  a.id[2] = c1 ? i1 : (c2 ? v : i2);
  a.sc[1] = c0 ? s0 : (c1 ? x : s1);
  a.id[1] = c0 ? i0 : (c1 ? v : i1);
  a.sc[0] = c0 ? x : s0;
  a.id[0] = c0 ? v : i0;
}

// Fold 16 consecutive columns v0 .. v0+15 (v0 a multiple of 16) of one row, of
// which the first nv (a multiple of 4) are vocabulary ids. c2s = log2(e) / T.
// Must be called by all 32 lanes of a warp together.
template <bool kSampling, bool kFull>
__device__ __forceinline__ void lm_fold16(LmAcc& a, const uint32_t (&raw)[16], int v0, int nv, float c2s,
                                          const PhiloxRow& pr, uint32_t k0, uint32_t k1, bool active) {
  if (kSampling) {
    // the chunk v0 / 16: its maximum, its mass relative to it, the row's LSE
    // partials, then one noise draw and one list entry for the whole chunk
    float lmax = __uint_as_float(raw[0]);
#pragma unroll
    for (int j = 1; j < 16; ++j)
      if (kFull || j < nv) lmax = fmaxf(lmax, __uint_as_float(raw[j]));
    const float cm = lmax * c2s;
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (kFull || j < nv) s += ex2_approx(fmaf(__uint_as_float(raw[j]), c2s, -cm));
    if (!active) return;
    const float mm = fmaxf(a.m, cm);
    a.s = a.s * ex2_approx(a.m - mm) + s * ex2_approx(cm - mm);
    a.m = mm;
    const uint32_t k = (uint32_t)v0 >> 4;
    const uint4 w = philox_row(k >> 2, pr, k0, k1);
    const uint32_t wk = (k & 2u) ? ((k & 1u) ? w.w : w.z) : ((k & 1u) ? w.y : w.x);
    topk_push_scan(a, cm + lg2_approx(s) - lg2_approx(neg_log2_u01(wk)), (int)k);
  } else {
    if (!active) return;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (kFull || j < nv) topk_push_scan(a, __uint_as_float(raw[j]), v0 + j);
  }
}

}  // namespace tc
}  // namespace dlite
