// select_budget.cu -- layer-level competitive budget (NestedKV technical
// summary, 3. Hoofd-gewijze Geheugentoewijzing; KV-cache survey blog §4.4,
// PyramidKV: the budget belongs to the layer, not to each head).
//
// Batch row b is one layer whose H heads share `budget` kept positions.  Every
// head keeps its sinks [0, S), its recent window [T-R, T) and its floor-S-R best
// middle positions (z descending, position ascending); the budget - H*floor
// slots left go to the best middle (head, position) pairs of the row not kept
// yet, in the order (z descending, head ascending, position ascending).
//
// Every pair gets a unique 64-bit key whose descending order is exactly that
// order: the order-preserving image of z in the high word and ~(h*T + position)
// in the low word.  A head's own order is the same key restricted to the head,
// so with
//   theta_h = the key of head h's (floor-S-R)-th best middle pair,
//   tau     = the key of the (budget-H*floor)-th best pair among the middle
//             pairs below their head's theta_h,
// head h keeps exactly its middle pairs with key >= min(theta_h, tau).
//
// One thread-block cluster per row; CTA c of the cluster owns heads c, c+CL, ...
//   1. floor: a radix select per owned head finds theta_h: 8-bit digits of the
//      64-bit key, most significant first, stopping as soon as the boundary
//      digit's bucket is taken whole (unique keys always stop by the 8th pass,
//      distinct scores by the 4th);
//   2. competition: the same radix select over the row's pool; each CTA
//      histograms its own heads and sums the cluster's histograms through
//      distributed shared memory, so every CTA takes the same decisions;
//   3. each CTA counts its heads' kept middle pairs (per warp, over a contiguous
//      range per warp) and stores the counts into every CTA of the cluster;
//      offsets are a prefix sum over heads;
//   4. each owned head writes its sinks, its kept middle positions (warp
//      ballots over the same ranges keep them ascending) and its recent window
//      at its offset.
// Integer work only after the key transform: the same z gives the same output.
#include <cooperative_groups.h>

#include "kvc_internal.cuh"
#include "select_common.cuh"

namespace cg = cooperative_groups;

namespace kvc {
namespace {

constexpr int NT = 1024;
constexpr int NW = NT / 32;
constexpr int kMaxCluster = 8;
constexpr int kMaxHeads = 256;
constexpr int kMaxOwned = kMaxHeads / kMaxCluster;  // heads per CTA when H > 8
constexpr uint64_t kNone = ~0ull;                   // above every key: selects nothing

struct Smem {
  RadixScratch<NT> rx;
  uint64_t theta[kMaxHeads];    // floor thresholds (owned heads' entries only)
  int cnt[kMaxHeads];           // kept positions per head, written by the owners
  int offs[kMaxHeads + 1];
  int wcnt[kMaxOwned][NW];      // kept middle pairs per (owned head, warp range)
};

// A head's middle range [0, n) split for 16-byte loads: `pre` scalars up to the
// first 16-byte boundary, n4 float4 vectors, then the scalars from `tail` on.
struct Split {
  int pre, n4, tail;
};
__device__ __forceinline__ Split split_of(const float *zm, int n) {
  const int mis = (int)((reinterpret_cast<uintptr_t>(zm) >> 2) & 3);
  Split sp;
  sp.pre = min(n, (4 - mis) & 3);
  sp.n4 = (n - sp.pre) >> 2;
  sp.tail = sp.pre + 4 * sp.n4;
  return sp;
}

// Calls f(key) for the middle pairs of one head, positions [S, S + n), with
// strided coalesced 16-byte loads, four in flight per thread (64 KB per CTA:
// enough to cover the latency of the repeated passes over L2).
template <typename F>
__device__ __forceinline__ void for_head(const float *__restrict__ zm, uint32_t flat0, int n, F &&f) {
  const Split sp = split_of(zm, n);
  const float4 *z4 = reinterpret_cast<const float4 *>(zm + sp.pre);
  for (int base = threadIdx.x; base < sp.n4; base += 4 * NT) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = base + u * NT;
      v[u] = (j < sp.n4) ? __ldg(z4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = base + u * NT;
      if (j < sp.n4) {
        const uint32_t i = flat0 + (uint32_t)(sp.pre + 4 * j);
        f(pair_key(v[u].x, i));
        f(pair_key(v[u].y, i + 1));
        f(pair_key(v[u].z, i + 2));
        f(pair_key(v[u].w, i + 3));
      }
    }
  }
  const int t = threadIdx.x, nt = n - sp.tail;
  if (t < sp.pre) f(pair_key(__ldg(zm + t), flat0 + (uint32_t)t));
  else if (t < sp.pre + nt) {
    const int i = sp.tail + (t - sp.pre);
    f(pair_key(__ldg(zm + i), flat0 + (uint32_t)i));
  }
}

__global__ __launch_bounds__(NT, 1) void select_budget_kernel(
    const float *__restrict__ z, int H, int T, int budget, int floor_k, int R, int S,
    int32_t *__restrict__ idx_out, int32_t *__restrict__ off_out) {
  __shared__ Smem sm;
  cg::cluster_group cl = cg::this_cluster();
  const int CL = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const long row = blockIdx.x / CL;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = T - R - S, nf = floor_k - R - S;
  const long long extra = (long long)budget - (long long)H * floor_k;
  const float *zrow = z + row * (long)H * T;
  auto zmid = [&](int h) { return zrow + (long)h * T + S; };
  auto flat0 = [&](int h) { return (uint32_t)h * (uint32_t)T + (uint32_t)S; };

  cl.sync();  // every CTA of the cluster is running before any remote access

  // 1. floor thresholds of the owned heads
  for (int h = rank; h < H; h += CL) {
    uint64_t th = kNone;
    if (nf > 0)
      th = radix_select_ge<NT, false>(sm.rx, nf, [&](auto &&f) { for_head(zmid(h), flat0(h), n, f); });
    if (threadIdx.x == 0) sm.theta[h] = th;
  }
  __syncthreads();

  // 2. competition over the middle pairs below their head's floor threshold
  uint64_t tau = kNone;
  if (extra > 0) {
    tau = radix_select_ge<NT, true>(sm.rx, (int)extra, [&](auto &&f) {
      for (int h = rank; h < H; h += CL) {
        const uint64_t th = sm.theta[h];
        for_head(zmid(h), flat0(h), n, [&](uint64_t key) {
          if (key < th) f(key);
        });
      }
    });
  }

  // 3. kept middle pairs per owned head and warp: warp 0 takes the scalars before
  // the first 16-byte boundary, every warp a contiguous run of float4 vectors,
  // the last warp the scalar tail; counts to every CTA of the cluster
  for (int h = rank, j = 0; h < H; h += CL, ++j) {
    const uint64_t lam = min(sm.theta[h], tau);
    const float *zm = zmid(h);
    const uint32_t f0 = flat0(h);
    const Split sp = split_of(zm, n);
    const float4 *z4 = reinterpret_cast<const float4 *>(zm + sp.pre);
    const int per4 = (sp.n4 + NW - 1) / NW;
    const int b0 = min(sp.n4, warp * per4), b1 = min(sp.n4, b0 + per4);
    int c = 0;
    if (warp == 0 && lane < sp.pre) c += pair_key(__ldg(zm + lane), f0 + (uint32_t)lane) >= lam;
#pragma unroll 4
    for (int q = b0 + lane; q < b1; q += 32) {
      const float4 v = __ldg(z4 + q);
      const uint32_t i = f0 + (uint32_t)(sp.pre + 4 * q);
      c += (pair_key(v.x, i) >= lam) + (pair_key(v.y, i + 1) >= lam) +
           (pair_key(v.z, i + 2) >= lam) + (pair_key(v.w, i + 3) >= lam);
    }
    if (warp == NW - 1 && lane < n - sp.tail)
      c += pair_key(__ldg(zm + sp.tail + lane), f0 + (uint32_t)(sp.tail + lane)) >= lam;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
    if (lane == 0) sm.wcnt[j][warp] = c;
    __syncthreads();
    if (threadIdx.x < CL) {
      int tot = 0;
      for (int w = 0; w < NW; ++w) tot += sm.wcnt[j][w];
      cl.map_shared_rank(&sm.cnt[0], threadIdx.x)[h] = S + R + tot;
    }
  }
  cl.sync();  // counts visible everywhere; the last remote access is above
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int h = 0; h < H; ++h) {
      sm.offs[h] = acc;
      acc += sm.cnt[h];
    }
    sm.offs[H] = acc;
  }
  __syncthreads();
  // The counts add up to the budget by construction; should they not, nothing
  // is written past the row: the offsets read -1 and no index is emitted.
  const bool consistent = sm.offs[H] == budget;
  if (rank == 0)
    for (int h = threadIdx.x; h <= H; h += NT)
      off_out[row * (H + 1) + h] = consistent ? sm.offs[h] : -1;
  if (!consistent) return;

  // 4. output, per owned head: sinks, kept middle positions ascending, recent
  int32_t *orow = idx_out + row * (long)budget;
  for (int h = rank, j = 0; h < H; h += CL, ++j) {
    int32_t *out = orow + sm.offs[h];
    const int kept_mid = sm.cnt[h] - S - R;
    for (int m = threadIdx.x; m < S; m += NT) out[m] = m;
    for (int m = threadIdx.x; m < R; m += NT) out[S + kept_mid + m] = T - R + m;
    int run = 0;
    for (int w = 0; w < warp; ++w) run += sm.wcnt[j][w];
    const uint64_t lam = min(sm.theta[h], tau);
    const float *zm = zmid(h);
    const uint32_t f0 = flat0(h);
    const Split sp = split_of(zm, n);
    const float4 *z4 = reinterpret_cast<const float4 *>(zm + sp.pre);
    const int per4 = (sp.n4 + NW - 1) / NW;
    const int b0 = min(sp.n4, warp * per4), b1 = min(sp.n4, b0 + per4);
    int32_t *mid = out + S;
    const unsigned below = (1u << lane) - 1u;
    if (warp == 0) {
      const bool keep = lane < sp.pre && pair_key(__ldg(zm + lane), f0 + (uint32_t)lane) >= lam;
      const unsigned m = __ballot_sync(0xFFFFFFFFu, keep);
      const int slot = run + __popc(m & below);
      if (keep && slot < kept_mid) mid[slot] = S + lane;
      run += __popc(m);
    }
    for (int q0 = b0; q0 < b1; q0 += 32) {
      const int q = q0 + lane;
      bool k0 = false, k1 = false, k2 = false, k3 = false;
      const int i = sp.pre + 4 * q;
      if (q < b1) {
        const float4 v = __ldg(z4 + q);
        const uint32_t fi = f0 + (uint32_t)i;
        k0 = pair_key(v.x, fi) >= lam;
        k1 = pair_key(v.y, fi + 1) >= lam;
        k2 = pair_key(v.z, fi + 2) >= lam;
        k3 = pair_key(v.w, fi + 3) >= lam;
      }
      const int c = (int)k0 + (int)k1 + (int)k2 + (int)k3;
      int incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += y;
      }
      int slot = run + incl - c;
      if (k0 && slot < kept_mid) mid[slot] = S + i;
      slot += k0;
      if (k1 && slot < kept_mid) mid[slot] = S + i + 1;
      slot += k1;
      if (k2 && slot < kept_mid) mid[slot] = S + i + 2;
      slot += k2;
      if (k3 && slot < kept_mid) mid[slot] = S + i + 3;
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (warp == NW - 1) {
      const int i = sp.tail + lane;
      const bool keep = i < n && pair_key(__ldg(zm + i), f0 + (uint32_t)i) >= lam;
      const unsigned m = __ballot_sync(0xFFFFFFFFu, keep);
      const int slot = run + __popc(m & below);
      if (keep && slot < kept_mid) mid[slot] = S + i;
    }
  }
}

}  // namespace

int launch_select_budget(const float *z, int B, int H, int T, int budget, int floor_k,
                         int recent, int sink, int32_t *idx, int32_t *off, cudaStream_t st) {
  const int CL = H < kMaxCluster ? H : kMaxCluster;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long)B * CL));
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)CL;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, select_budget_kernel, z, H, T, budget, floor_k,
                                           recent, sink, idx, off);
  if (e != cudaSuccess) return cuda_failure(e, "budget selection kernel");
  return launch_status();
}

}  // namespace kvc
