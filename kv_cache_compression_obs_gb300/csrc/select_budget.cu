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
//   1. floor: per owned head, a histogram of the keys' top 12 bits (one stream
//      over the head's scores) finds the bin holding theta_h; a second stream
//      gathers that bin's keys on chip, and a radix select over them alone
//      (8-bit digits, most significant first, stopping as soon as the boundary
//      digit's bucket is taken whole) gives theta_h exactly.  A bin too large
//      to gather (heavy ties) falls back to the radix select over the streamed
//      head;
//   2. competition: the same two streams over the row's pool, the histograms
//      summed over the cluster through distributed shared memory (every CTA
//      reads every histogram and takes the same decisions), then the radix
//      select over the cluster's gathered boundary-bin keys (histograms summed
//      through distributed shared memory), with the same fallback;
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

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int kMaxCluster = 8;
constexpr int kMaxHeads = 256;
constexpr int kMaxOwned = kMaxHeads / kMaxCluster;  // heads per CTA when H > 8
constexpr uint64_t kNone = ~0ull;                   // above every key: selects nothing
constexpr int kBins = 4096;                         // first digit: the key's top 12 bits
constexpr int kBinShift = 64 - 12;
constexpr int kListCap = 4096;                      // boundary-bin candidates held on chip

struct Smem {
  RadixScratch<NT> rx;
  uint64_t theta[kMaxHeads];    // floor thresholds (owned heads' entries only)
  int cnt[kMaxHeads];           // kept positions per head, written by the owners
  int offs[kMaxHeads + 1];
  int wcnt[kMaxOwned][NW];      // kept middle pairs per (owned head, warp range)
  int wsum[NW];
  int bin, need, above, list_n, overflow;
};

// Dynamic shared memory: the first-digit histogram and the boundary bin's
// candidate keys (the list region also holds the cluster's summed histogram).
struct Dyn {
  uint32_t hist[kBins];
  uint64_t list[kListCap];
};
static_assert(sizeof(uint64_t) * kListCap >= sizeof(uint32_t) * kBins, "summed histogram fits the list");

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
// strided coalesced 16-byte loads, four in flight per thread (32 KB per CTA,
// two CTAs per SM).
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

// In a histogram of kBins counts (bins taken from the top), the bin where the
// count of keys in it or above first reaches `need`: sm.bin, sm.need (how many of
// that bin's keys are needed) and sm.above.  Every thread of the CTA must call.
__device__ void find_boundary(const uint32_t *h, int need, Smem &sm) {
  constexpr int PER = kBins / NT;
  const int t = threadIdx.x;
  int mine = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) mine += (int)h[kBins - 1 - PER * t - i];
  int total;
  const int before = block_exclusive_scan<NT>(mine, sm.wsum, &total);
  if (before < need && need <= before + mine) {
    int acc = before;
    for (int i = 0; i < PER; ++i) {
      const int b = kBins - 1 - PER * t - i;
      const int c = (int)h[b];
      if (need <= acc + c) {
        sm.bin = b;
        sm.need = need - acc;
        sm.above = acc;
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

__global__ __launch_bounds__(NT, 2) void select_budget_kernel(
    const float *__restrict__ z, int H, int T, int budget, int floor_k, int R, int S,
    int32_t *__restrict__ idx_out, int32_t *__restrict__ off_out) {
  __shared__ Smem sm;
  extern __shared__ __align__(16) unsigned char dyn_raw[];
  Dyn &dy = *reinterpret_cast<Dyn *>(dyn_raw);
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

  // 1. floor thresholds of the owned heads.  Two streams over the head: a
  // histogram of the keys' top 12 bits finds the boundary bin, then the bin's
  // keys (a few hundred for spread-out scores) are gathered on chip and the
  // radix select runs over them alone.  A bin too large to gather (heavy ties)
  // takes the radix select over the streamed head instead.
  for (int h = rank; h < H; h += CL) {
    uint64_t th = kNone;
    if (nf > 0) {
      for (int e = threadIdx.x; e < kBins; e += NT) dy.hist[e] = 0u;
      __syncthreads();
      for_head(zmid(h), flat0(h), n, [&](uint64_t key) { atomicAdd(&dy.hist[key >> kBinShift], 1u); });
      __syncthreads();
      find_boundary(dy.hist, nf, sm);
      const int b = sm.bin, need = sm.need;
      if (dy.hist[b] <= (uint32_t)kListCap) {
        if (threadIdx.x == 0) sm.list_n = 0;
        __syncthreads();
        for_head(zmid(h), flat0(h), n, [&](uint64_t key) {
          if ((int)(key >> kBinShift) == b) dy.list[atomicAdd(&sm.list_n, 1)] = key;
        });
        __syncthreads();
        const int ln = sm.list_n;
        th = radix_select_ge<NT, false>(sm.rx, need, [&](auto &&f) {
          for (int i = threadIdx.x; i < ln; i += NT) f(dy.list[i]);
        });
        // the select stops at the first digit that settles the list; the lower
        // bins' keys must stay below the threshold too
        th = max(th, (uint64_t)b << kBinShift);
      } else {
        th = radix_select_ge<NT, false>(sm.rx, nf, [&](auto &&f) { for_head(zmid(h), flat0(h), n, f); });
      }
    }
    if (threadIdx.x == 0) sm.theta[h] = th;
    __syncthreads();  // the histogram and the list serve the next head
  }

  // 2. competition over the middle pairs below their head's floor threshold: the
  // same two streams, the histograms summed over the cluster (every CTA reads
  // every CTA's histogram and takes the same decisions); the radix select then
  // runs over the cluster's gathered boundary-bin keys
  uint64_t tau = kNone;
  if (extra > 0) {
    for (int e = threadIdx.x; e < kBins; e += NT) dy.hist[e] = 0u;
    __syncthreads();
    for (int h = rank; h < H; h += CL) {
      const uint64_t th = sm.theta[h];
      for_head(zmid(h), flat0(h), n, [&](uint64_t key) {
        if (key < th) atomicAdd(&dy.hist[key >> kBinShift], 1u);
      });
    }
    cl.sync();  // every histogram of the cluster is complete
    uint32_t *gs = reinterpret_cast<uint32_t *>(dy.list);  // the cluster's sum, in the list region
    for (int e = threadIdx.x; e < kBins; e += NT) {
      uint32_t g = 0;
      for (int r = 0; r < CL; ++r) g += cl.map_shared_rank(dy.hist, r)[e];
      gs[e] = g;
    }
    __syncthreads();
    find_boundary(gs, (int)extra, sm);
    const int b = sm.bin, need = sm.need;
    if (threadIdx.x == 0) {
      int ovf = 0;
      for (int r = 0; r < CL; ++r) ovf |= cl.map_shared_rank(dy.hist, r)[b] > (uint32_t)kListCap;
      sm.overflow = ovf;
      sm.list_n = 0;
    }
    __syncthreads();
    if (!sm.overflow) {
      for (int h = rank; h < H; h += CL) {
        const uint64_t th = sm.theta[h];
        for_head(zmid(h), flat0(h), n, [&](uint64_t key) {
          if (key < th && (int)(key >> kBinShift) == b) dy.list[atomicAdd(&sm.list_n, 1)] = key;
        });
      }
      __syncthreads();
      const int ln = sm.list_n;
      tau = radix_select_ge<NT, true>(sm.rx, need, [&](auto &&f) {
        for (int i = threadIdx.x; i < ln; i += NT) f(dy.list[i]);
      });
      tau = max(tau, (uint64_t)b << kBinShift);  // as for the floor thresholds
    } else {
      tau = radix_select_ge<NT, true>(sm.rx, (int)extra, [&](auto &&f) {
        for (int h = rank; h < H; h += CL) {
          const uint64_t th = sm.theta[h];
          for_head(zmid(h), flat0(h), n, [&](uint64_t key) {
            if (key < th) f(key);
          });
        }
      });
    }
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
  cfg.dynamicSmemBytes = sizeof(Dyn);
  cfg.stream = st;
  if (ensure_smem((const void *)select_budget_kernel, sizeof(Dyn)))
    return cuda_failure(cudaErrorInvalidValue, "budget selection kernel: shared memory");
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
