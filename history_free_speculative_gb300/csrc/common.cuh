// Shared device helpers of the DLite CUDA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dlite {

typedef __nv_bfloat16 bf16;

// Sticky device status bits (mirrors DLITE_DEV_* in dlite.h).
constexpr int kDevTimeout = 1;
constexpr int kDevBounds = 2;

__device__ __forceinline__ void flag_status(int* st, int bits) {
  if (st) atomicOr(st, bits);
}

// ---------------------------------------------------------------- conversions

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }

// Two-plane bf16 representation of an fp32 value: hi = rn(x), lo = rn(x - hi).
__device__ __forceinline__ void split_bf16(float x, bf16& hi, bf16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// ---------------------------------------------------------------- tiled weights
// Weight matrices that feed the tensor-core products are stored as 64 x 64
// tiles: element (r, c) of a [rows, cols] matrix (rows padded to a multiple of
// 64, cols a multiple of 64) sits at tile (r/64, c/64), tiles ordered row-tile
// major, each tile 64 rows x 64 columns row-major. One k block (64 columns) of
// a 64-row slab is then one contiguous 8 KB chunk, so a CTA streams its slab
// from HBM as long sequential runs.
__host__ __device__ __forceinline__ size_t tiled_index(size_t r, size_t c, size_t cols) {
  return ((r >> 6) * (cols >> 6) + (c >> 6)) * 4096 + (r & 63) * 64 + (c & 63);
}

// ---------------------------------------------------------------- Philox4x32-10
// Salmon, Moraes, Dror & Shaw, "Parallel random numbers: as easy as 1, 2, 3"
// (SC'11): ten rounds of the 4x32 Philox S-box with the key bumped by the two
// Weyl constants between rounds.
constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

constexpr uint32_t kTagGumbel = 1;
constexpr uint32_t kTagAccept = 2;
constexpr uint32_t kTagResid = 3;
constexpr uint32_t kTagBonus = 4;
constexpr uint32_t kTagPick = 8;  // the draw inside the chosen vocabulary chunk
constexpr int kChunk = 16;        // vocabulary ids per chunk of the two-level draft draw
constexpr int kProposals = 32;

__device__ __forceinline__ uint4 philox(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                        uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += kPhiloxW0;
      k1 += kPhiloxW1;
    }
    // one 32x32 -> 64-bit multiply gives both halves of each product
    const uint64_t p0 = (uint64_t)kPhiloxM0 * c0;
    const uint64_t p1 = (uint64_t)kPhiloxM1 * c2;
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return make_uint4(c0, c1, c2, c3);
}

// Uniform in (0,1) from the top 23 bits; exact in fp32 and fp64.
__device__ __forceinline__ float u01f(uint32_t x) {
  return ((float)(x >> 9) + 0.5f) * 1.1920928955078125e-07f;
}
__device__ __forceinline__ double u01d(uint32_t x) {
  return ((double)(x >> 9) + 0.5) * 1.1920928955078125e-07;
}

// ---------------------------------------------------------------- programmatic dependent launch
// Kernels of the round are launched with programmatic stream serialization:
// a kernel may begin while its predecessor drains. pdl_trigger lets the next
// kernel launch; pdl_wait blocks until the predecessor has completed and its
// writes are visible, and must precede any access to data a predecessor
// produces or consumes.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum (blockDim.x multiple of 32, <= 1024). `red` holds >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  float t = (threadIdx.x < nw) ? red[threadIdx.x] : 0.f;
  if (wid == 0) t = warp_sum(t);
  if (threadIdx.x == 0) red[0] = t;
  __syncthreads();
  return red[0];
}

}  // namespace dlite
