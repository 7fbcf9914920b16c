// select_common.cuh -- integer helpers shared by the two selection kernels.
#pragma once

#include <cstdint>

namespace kvc {

// Monotone map float -> uint32 (larger float, larger key); -0.0 maps like +0.0.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide prefix sum of one int per thread of an NT-thread block;
// *total gets the sum.  warp_sums holds NT/32 ints; every thread must call.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < NW) ? warp_sums[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, off);
      if (lane >= off) w += y;
    }
    if (lane < NW) warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0) ? warp_sums[warp - 1] : 0;
  *total = warp_sums[NW - 1];
  __syncthreads();  // warp_sums is reused by the next call
  return before + x - v;
}

}  // namespace kvc
