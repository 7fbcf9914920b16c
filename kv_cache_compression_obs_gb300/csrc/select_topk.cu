// select_topk.cu -- budgeted per-head Top-K with a protected recent window.
//
// H2O page, 双缓冲 and 为什么要按头独立驱逐: every head keeps the last R
// positions and the k - R best of [0, T - R) in the order (z descending,
// position ascending); the kept positions are written in ascending order.
// With S sinks (KV-cache survey blog §4.1-4.2) the first S positions are kept
// too and the heavy part is the k - R - S best of [S, T - R).
//
// One 1024-thread block per head:
//   1. exact radix select (4 passes of 8 bits over order-preserving uint32
//      keys, per-warp shared-memory histograms) finds the (k-R)-th largest key u*
//      and how many of the keys equal to u* must be taken;
//   2. one ordered pass keeps every key > u* and the first `need` keys == u*
//      (block-wide scans give each kept position its output slot), so the
//      positions come out ascending without a sort;
//   3. the recent window is appended.
// Integer work only after the key transform: the same z always gives the same idx.
#include "kvc_internal.cuh"
#include "select_common.cuh"

namespace kvc {
namespace {

constexpr int NT = 1024;
constexpr int NW = NT / 32;

__global__ __launch_bounds__(NT) void select_topk_kernel(const float *__restrict__ z, int T,
                                                         int k, int R, int S,
                                                         int32_t *__restrict__ idx_out) {
  __shared__ uint32_t hist[NW][256];
  __shared__ uint32_t tot[256];
  __shared__ int warp_sums[NW];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_need;
  const long head = blockIdx.x;
  const float *zv = z + head * (long)T + S;  // candidates [S, T - R), indexed from S
  int32_t *out = idx_out + head * (long)k;
  const int n = T - R - S;   // candidates
  const int nh = k - R - S;  // heavy slots
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  if (nh >= n) {  // k == T: everything is kept
    for (int m = threadIdx.x; m < k; m += NT) out[m] = m;
    return;
  }
  for (int m = threadIdx.x; m < S; m += NT) out[m] = m;  // the sinks, first
  out += S;

  uint32_t prefix = 0, mask = 0;
  int need = nh;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int e = threadIdx.x; e < NW * 256; e += NT) (&hist[0][0])[e] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += NT) {
      const uint32_t u = order_key(zv[i]);
      if ((u & mask) == prefix) atomicAdd(&hist[warp][(u >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 256) {
      uint32_t t = 0;
      for (int w = 0; w < NW; ++w) t += hist[w][threadIdx.x];
      tot[threadIdx.x] = t;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns digits 255-8l .. 248-8l (descending)
      uint32_t mine = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) mine += tot[255 - 8 * lane - i];
      uint32_t incl = mine;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += y;
      }
      uint32_t above = incl - mine;  // count in digits above this lane's range
      if (above < (uint32_t)need && (uint32_t)need <= incl) {
#pragma unroll 1
        for (int i = 0; i < 8; ++i) {
          const int dgt = 255 - 8 * lane - i;
          const uint32_t c = tot[dgt];
          if ((uint32_t)need <= above + c) {
            sh_prefix = prefix | ((uint32_t)dgt << shift);
            sh_need = need - (int)above;
            break;
          }
          above += c;
        }
      }
    }
    __syncthreads();
    prefix = sh_prefix;
    need = sh_need;
    mask |= 255u << shift;
    __syncthreads();
  }

  // ordered keep pass: keys > u*, and the first `need` keys == u*
  const uint32_t ustar = prefix;
  int carry_eq = 0, carry_keep = 0;
  for (int base = 0; base < n; base += NT) {
    const int i = base + threadIdx.x;
    const uint32_t u = (i < n) ? order_key(zv[i]) : 0u;
    const int gt = (i < n) && (u > ustar);
    const int eq = (i < n) && (u == ustar);
    int eq_total, keep_total;
    const int eq_rank = carry_eq + block_exclusive_scan<NT>(eq, warp_sums, &eq_total);
    const int keep = gt || (eq && eq_rank < need);
    const int slot = carry_keep + block_exclusive_scan<NT>(keep, warp_sums, &keep_total);
    if (keep && slot < nh) out[slot] = S + i;
    carry_eq += eq_total;
    carry_keep += keep_total;
  }
  for (int m = threadIdx.x; m < R; m += NT) out[nh + m] = S + n + m;
  (void)lane;
}

}  // namespace

int launch_select_topk(const float *z, int B, int H, int T, int k, int recent, int sink,
                       int32_t *idx, cudaStream_t st) {
  const long heads = (long)B * H;
  select_topk_kernel<<<(unsigned)heads, NT, 0, st>>>(z, T, k, recent, sink, idx);
  return launch_status();
}

}  // namespace kvc
