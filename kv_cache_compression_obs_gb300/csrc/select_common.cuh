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

#include <cooperative_groups.h>
#include <cstddef>
#include <type_traits>

namespace kvc {

// Scratch of radix_select_ge for an NT-thread block; warp w counts into
// histogram copy w % HC (HC a power of two dividing the warps: fewer copies, less
// shared memory, more atomics on one copy).
template <int NT, int HC = NT / 32>
struct RadixScratch {
  static constexpr int NW = NT / 32;
  static constexpr int NH = HC;
  static_assert((HC & (HC - 1)) == 0 && NW % HC == 0, "histogram copies must divide the warps");
  uint32_t hist[HC][256];  // histogram copies
  uint32_t tot[2][256];    // this CTA's histogram of a pass (read by the cluster)
  uint32_t gsum[256];      // the (cluster's) histogram of a pass
  uint64_t sh_prefix;
  int sh_need, sh_done;
};

// Warp 0 of the block: in a 256-digit histogram h taken from the top, the digit
// where the count at or above it first reaches `need`.  Writes sm.sh_prefix
// (prefix with that digit at `shift`), sm.sh_need (how many of the digit's keys
// are needed) and sm.sh_done (whether that is all of them).
template <typename Scratch>
__device__ __forceinline__ void digit_boundary(const uint32_t *h, int need, uint64_t prefix, int shift,
                                               Scratch &sm) {
  const int lane = threadIdx.x & 31;
  uint32_t mine = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) mine += h[255 - 8 * lane - i];  // lane l: digits 255-8l .. 248-8l
  uint32_t incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += y;
  }
  uint32_t above = incl - mine;
  if (above < (uint32_t)need && (uint32_t)need <= incl) {
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      const int dgt = 255 - 8 * lane - i;
      const uint32_t c = h[dgt];
      if ((uint32_t)need <= above + c) {
        sm.sh_prefix = prefix | ((uint64_t)dgt << shift);
        sm.sh_need = need - (int)above;
        sm.sh_done = ((uint32_t)need == above + c);
        break;
      }
      above += c;
    }
  }
}

// Threshold thr such that exactly `need` candidate keys are >= thr, for unique
// 64-bit keys and 1 <= need <= number of candidates.  visit(f) calls f(key) for
// every candidate key this thread owns.  8-bit digits, most significant first;
// the search stops as soon as the boundary digit's bucket is taken whole (at
// the last digit unique keys always fill it exactly).  CLUSTER: the candidates
// are spread over the cluster's CTAs, each histogramming its own and summing
// all of them through distributed shared memory, so every CTA takes the same
// decisions and runs the same passes.  Every thread of every CTA must call.
//
// visit_hi (optional): visit_hi(f) calls f(key >> 32) for every candidate; the
// four passes over the high word then use 32-bit keys.  pass0_filled: the caller
// has already histogrammed the top byte (key >> 56) into sm.hist (per warp).
template <int NT, bool CLUSTER, typename Visit, typename VisitHi = std::nullptr_t, int HC = NT / 32>
__device__ uint64_t radix_select_ge(RadixScratch<NT, HC> &sm, int need, Visit visit,
                                    VisitHi visit_hi = nullptr, bool pass0_filled = false) {
  const int hw = (threadIdx.x >> 5) & (HC - 1);  // this warp's histogram copy
  constexpr bool HI32 = !std::is_same<VisitHi, std::nullptr_t>::value;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t prefix = 0, hmask = 0;
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    const int buf = pass & 1;
    if (!(pass == 0 && pass0_filled)) {
      if (pass == 0) {  // later passes find the histograms zeroed by the previous reduction
        for (int e = threadIdx.x; e < HC * 256; e += NT) (&sm.hist[0][0])[e] = 0u;
        __syncthreads();
      }
      bool done_hi = false;
      if constexpr (HI32) {
        if (shift >= 32) {
          const uint32_t p32 = (uint32_t)(prefix >> 32), m32 = (uint32_t)(hmask >> 32);
          const int sh = shift - 32;
          visit_hi([&](uint32_t k) {
            if ((k & m32) == p32) atomicAdd(&sm.hist[hw][(k >> sh) & 255u], 1u);
          });
          done_hi = true;
        }
      }
      if (!done_hi)
        visit([&](uint64_t key) {
          if ((key & hmask) == prefix) atomicAdd(&sm.hist[hw][(uint32_t)(key >> shift) & 255u], 1u);
        });
    }
    __syncthreads();
    for (int d = threadIdx.x; d < 256; d += NT) {
      uint32_t t = 0;
#pragma unroll 8
      for (int w = 0; w < HC; ++w) {
        t += sm.hist[w][d];
        sm.hist[w][d] = 0u;  // ready for the next pass (barriers follow before its visit)
      }
      sm.tot[buf][d] = t;
    }
    if constexpr (CLUSTER) {
      // tot[buf] is rewritten two passes later, after the next cluster barrier,
      // by which time every CTA has finished reading it.
      cooperative_groups::cluster_group cl = cooperative_groups::this_cluster();
      cl.sync();
      const unsigned ncl = cl.num_blocks();
      for (int d = threadIdx.x; d < 256; d += NT) {
        uint32_t g = 0;
#pragma unroll
        for (unsigned r = 0; r < 8; ++r)  // independent remote loads, all in flight
          if (r < ncl) g += cl.map_shared_rank(&sm.tot[buf][0], r)[d];
        for (unsigned r = 8; r < ncl; ++r) g += cl.map_shared_rank(&sm.tot[buf][0], r)[d];
        sm.gsum[d] = g;
      }
    } else {
      for (int d = threadIdx.x; d < 256; d += NT) sm.gsum[d] = sm.tot[buf][d];
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns digits 255-8l .. 248-8l (descending)
      uint32_t mine = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) mine += sm.gsum[255 - 8 * lane - i];
      uint32_t incl = mine;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += y;
      }
      uint32_t above = incl - mine;
      if (above < (uint32_t)need && (uint32_t)need <= incl) {
#pragma unroll 1
        for (int i = 0; i < 8; ++i) {
          const int dgt = 255 - 8 * lane - i;
          const uint32_t c = sm.gsum[dgt];
          if ((uint32_t)need <= above + c) {
            sm.sh_prefix = prefix | ((uint64_t)dgt << shift);
            sm.sh_need = need - (int)above;
            sm.sh_done = ((uint32_t)need == above + c);
            break;
          }
          above += c;
        }
      }
    }
    __syncthreads();
    prefix = sm.sh_prefix;
    need = sm.sh_need;
    const int done = sm.sh_done;
    hmask |= 255ull << shift;
    __syncthreads();  // sh_* and gsum are rewritten by the next pass
    if (done) break;
  }
  return prefix;
}

// Unique 64-bit selection key of element `flat`: the order-preserving image of z
// in the high word, ~flat in the low word, so that descending keys are
// (z descending, flat ascending).
__device__ __forceinline__ uint64_t pair_key(float z, uint32_t flat) {
  return ((uint64_t)order_key(z) << 32) | (uint64_t)(0xFFFFFFFFu - flat);
}
__device__ __forceinline__ uint64_t pair_key_u(uint32_t okey, uint32_t flat) {
  return ((uint64_t)okey << 32) | (uint64_t)(0xFFFFFFFFu - flat);
}

}  // namespace kvc
