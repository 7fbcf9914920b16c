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

__device__ __forceinline__ uint64_t pair_key(float z, uint32_t flat) {
  return ((uint64_t)order_key(z) << 32) | (uint64_t)(0xFFFFFFFFu - flat);
}

struct Smem {
  uint32_t hist[NW][256];
  uint32_t tot[2][256];         // this CTA's histogram of a pass, read by the cluster
  uint32_t gsum[256];           // the cluster's histogram of a pass
  uint64_t theta[kMaxHeads];    // floor thresholds (owned heads' entries only)
  int cnt[kMaxHeads];           // kept positions per head, written by the owners
  int offs[kMaxHeads + 1];
  int wcnt[kMaxOwned][NW];      // kept middle pairs per (owned head, warp range)
  uint64_t sh_prefix;
  int sh_need, sh_done;
};

// Threshold thr such that exactly `need` candidate keys are >= thr, for unique
// keys and 1 <= need <= number of candidates.  visit(f) calls f(key) for every
// candidate key this thread owns.  CLUSTER: the candidates are spread over the
// cluster's CTAs, each histogramming its own; every CTA reads the others'
// histograms and takes the same decision, so all run the same passes.
template <bool CLUSTER, typename Visit>
__device__ uint64_t radix_select(Smem &sm, int need, Visit visit) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t prefix = 0, hmask = 0;
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    const int buf = pass & 1;
    for (int e = threadIdx.x; e < NW * 256; e += NT) (&sm.hist[0][0])[e] = 0u;
    __syncthreads();
    visit([&](uint64_t key) {
      if ((key & hmask) == prefix) atomicAdd(&sm.hist[warp][(uint32_t)(key >> shift) & 255u], 1u);
    });
    __syncthreads();
    if (threadIdx.x < 256) {
      uint32_t t = 0;
#pragma unroll 8
      for (int w = 0; w < NW; ++w) t += sm.hist[w][threadIdx.x];
      sm.tot[buf][threadIdx.x] = t;
    }
    if constexpr (CLUSTER) {
      // tot[buf] is rewritten two passes later, after the next cluster barrier,
      // by which time every CTA has finished reading it.
      cg::cluster_group cl = cg::this_cluster();
      cl.sync();
      if (threadIdx.x < 256) {
        uint32_t g = 0;
        for (unsigned r = 0; r < cl.num_blocks(); ++r)
          g += cl.map_shared_rank(&sm.tot[buf][0], r)[threadIdx.x];
        sm.gsum[threadIdx.x] = g;
      }
    } else {
      if (threadIdx.x < 256) sm.gsum[threadIdx.x] = sm.tot[buf][threadIdx.x];
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
  return prefix;  // at the last digit unique keys fill the boundary bucket exactly
}

// Calls f(key) for the middle pairs of one head, positions [S, S + n), with
// strided coalesced loads, four in flight per thread.
template <typename F>
__device__ __forceinline__ void for_head(const float *__restrict__ zm, uint32_t flat0, int n, F &&f) {
  for (int base = threadIdx.x; base < n; base += 4 * NT) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * NT;
      v[u] = (i < n) ? __ldg(zm + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = base + u * NT;
      if (i < n) f(pair_key(v[u], flat0 + (uint32_t)i));
    }
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
      th = radix_select<false>(sm, nf, [&](auto &&f) { for_head(zmid(h), flat0(h), n, f); });
    if (threadIdx.x == 0) sm.theta[h] = th;
  }
  __syncthreads();

  // 2. competition over the middle pairs below their head's floor threshold
  uint64_t tau = kNone;
  if (extra > 0) {
    tau = radix_select<true>(sm, (int)extra, [&](auto &&f) {
      for (int h = rank; h < H; h += CL) {
        const uint64_t th = sm.theta[h];
        for_head(zmid(h), flat0(h), n, [&](uint64_t key) {
          if (key < th) f(key);
        });
      }
    });
  }

  // 3. kept middle pairs per owned head and warp range; counts to every CTA
  const int per = ((n + NW - 1) / NW + 31) & ~31;
  const int lo = min(n, warp * per), hi = min(n, lo + per);
  for (int h = rank, j = 0; h < H; h += CL, ++j) {
    const uint64_t lam = min(sm.theta[h], tau);
    const float *zm = zmid(h);
    const uint32_t f0 = flat0(h);
    int c = 0;
#pragma unroll 4
    for (int i = lo + lane; i < hi; i += 32) c += pair_key(__ldg(zm + i), f0 + (uint32_t)i) >= lam;
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
    int32_t *mid = out + S;
    for (int i0 = lo; i0 < hi; i0 += 32) {
      const int i = i0 + lane;
      const bool keep = i < hi && pair_key(__ldg(zm + i), f0 + (uint32_t)i) >= lam;
      const unsigned m = __ballot_sync(0xFFFFFFFFu, keep);
      if (keep) mid[run + __popc(m & ((1u << lane) - 1u))] = S + i;
      run += __popc(m);
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
