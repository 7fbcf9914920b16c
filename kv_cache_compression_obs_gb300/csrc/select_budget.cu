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
// Scores concentrate: a head's threshold bin of the keys' top 12 bits can hold
// thousands of pairs and the competition's tens of thousands, so both
// thresholds are found through a bucket of the keys' top 20 bits (a 12-bit
// histogram, then an 8-bit one inside the boundary bin), whose pairs (tens to
// hundreds) are gathered on chip for an exact radix select.
//
// One thread-block cluster per row; CTA c of the cluster owns heads c, c+CL, ...
// Up to three streams over each owned head's scores, then the output:
//   0. (one head per CTA) a sample of every 16th vector predicts theta_h's bin
//      and, summed over the cluster, tau's bin;
//   1. the 12-bit histogram (and the second digits of the predicted bins):
//      theta_h's bin and how many of its pairs reach theta_h.  The
//      competition's 12-bit histogram (pairs below theta_h) follows from these
//      counts alone; summed over the cluster through distributed shared memory
//      it gives tau's bin;
//   2. the second digits of theta_h's bin, and of tau's bin where that lies
//      below theta_h's (where the two bins are one, the competition's digits
//      follow from theta_h's), streamed only where step 1 did not take them;
//      summed over the cluster they give tau's bucket;
//   3. the gather of theta_h's bucket and of tau's bucket, counting per warp
//      range the pairs above each and recording in a shared-memory bitmask the
//      pairs above the lower of the two buckets (kept whatever the thresholds);
//      theta_h follows from its bucket's pairs, then tau from the cluster's
//      gathered pairs below their head's theta, read in place through
//      distributed shared memory.  The kept middle pairs per (owned head, warp
//      range) follow from the counts (head limited by theta_h, or by tau); they
//      go to every CTA, and offsets are a prefix sum over heads; the kept pairs
//      of the threshold's own bucket are marked in the bitmask from its list;
//   4. output: each owned head writes its sinks, its kept middle positions
//      (from the bitmask, ascending over the same warp ranges) and its recent
//      window at its offset.
// A bucket too large to gather (heavy ties) falls back to a radix select over
// the streamed pairs, the kept counts to a counting stream and the output to a
// stream with warp ballots.
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
constexpr int kSubShift = kBinShift - 8;            // second digit; a bucket is the top 20 bits
constexpr int kListCap = 2048;                      // bucket pairs held on chip per CTA
constexpr int kGroups = 64;                         // groups of kBins / kGroups bins (tau's bin)
constexpr int kBmWords = 8200;                      // kept-pair bitmasks of the owned heads
                                                    // (a 128K-position head takes 4098 words)

struct Smem {
  RadixScratch<NT> rx;
  uint64_t theta[kMaxHeads];   // floor thresholds of every head of the row (pushed by owners)
  int cnt[kMaxHeads];          // kept positions per head, written by the owners
  int offs[kMaxHeads + 1];
  int wcnt[kMaxOwned][NW];     // kept middle pairs per (owned head, warp range)
  int wth[kMaxOwned][NW];      // middle pairs >= theta_h per (owned head, warp range)
  int wtau[kMaxOwned][NW];     // middle pairs above tau's bucket per (owned head, warp range)
  int thok[kMaxOwned];         // wth holds the counts
  int b1[kMaxOwned];           // theta_h's 12-bit bin (kBins: no floor)
  int need1[kMaxOwned];        // pairs of that bin at or above theta_h
  uint32_t p20h[kMaxOwned];    // theta_h's 20-bit bucket (~0u: none gathered)
  int need2[kMaxOwned];        // pairs of that bucket at or above theta_h
  int big[kMaxOwned];          // the bucket is too large to gather
  int bmok[kMaxOwned];         // the head's kept pairs are in its bitmask
  int nonneg[kMaxOwned];       // the head holds no negative score
  uint32_t h8[512];            // second digits: of theta_h's bin [0, 256), and this
                               // CTA's of tau's bin (competition) [256, 512)
  uint32_t g8[256];            // the cluster's sum of them
  uint32_t h256[256];          // digit histogram of the selects inside a bucket
  uint32_t ccoarse[kGroups];   // this CTA's competition counts per group of bins (read by the cluster)
  uint32_t wsub[6][256];       // second digits of the predicted bins, taken by the first stream
  int wsum[NW];
  int lnr[kMaxCluster];        // competition bucket pairs held per CTA (pushed)
  int ovr[kMaxCluster];        // competition bucket overflowed per CTA (pushed)
  int bin, need, above, list_n, tl_n, red;
};

// Dynamic shared memory.  Steps 1-2: the 12-bit histogram of one head (then the
// cluster's summed competition histogram) and the competition's 12-bit
// histogram of this CTA (read by the cluster).  Step 3 on: the same bytes hold
// the gathered pairs of one head's floor bucket and of the competition's bucket.
union Dyn {
  struct {
    uint32_t hist[kBins];
    uint32_t comp[kBins];
  } h;
  struct {
    uint64_t tlist[kListCap];
    uint64_t clist[kListCap];
  } l;
};
static_assert(sizeof(uint64_t) * kListCap == sizeof(uint32_t) * kBins, "lists overlay the histograms");

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

// Warp ranges of a head: warp 0 takes the scalars before the first 16-byte
// boundary, every warp a contiguous run of per4 float4 vectors, the last warp
// the scalar tail.  The warp whose range holds middle position i:
__device__ __forceinline__ int warp_of(int i, const Split &sp, int per4) {
  if (i < sp.pre) return 0;
  if (i >= sp.tail) return NW - 1;
  return ((i - sp.pre) >> 2) / per4;
}

// The order key; NONNEG: the head holds no negative score (-0 aside), so the
// key is the bit pattern with the sign bit set (the same value, one instruction).
template <bool NONNEG>
__device__ __forceinline__ uint32_t okey(float f) {
  return NONNEG ? (__float_as_uint(f) | 0x80000000u) : order_key(f);
}

// A pair's order key (the high word of its 64-bit key) and its flat index
// h*T + position; the streams pass these, and the 64-bit key is formed only
// where a pair is kept in a list.  Comparisons against a 64-bit threshold:
__device__ __forceinline__ bool key_ge(uint32_t ok, uint32_t flat, uint64_t thr) {
  const uint32_t th = (uint32_t)(thr >> 32);
  return ok > th || (ok == th && 0xFFFFFFFFu - flat >= (uint32_t)thr);
}
constexpr int kBinShift32 = kBinShift - 32;  // the bins and buckets on the order key
constexpr int kSubShift32 = kSubShift - 32;

// Calls f(order key, flat index) for the middle pairs of one head, positions
// [S, S + n), with strided coalesced 16-byte loads, eight in flight per thread.
template <bool NONNEG = false, typename F>
__device__ __forceinline__ void for_head(const float *__restrict__ zm, uint32_t flat0, int n, F &&f) {
  const Split sp = split_of(zm, n);
  const float4 *z4 = reinterpret_cast<const float4 *>(zm + sp.pre);
  for (int base = threadIdx.x; base < sp.n4; base += 8 * NT) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = base + u * NT;
      v[u] = (j < sp.n4) ? __ldg(z4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = base + u * NT;
      if (j < sp.n4) {
        const uint32_t i = flat0 + (uint32_t)(sp.pre + 4 * j);
        f(okey<NONNEG>(v[u].x), i);
        f(okey<NONNEG>(v[u].y), i + 1);
        f(okey<NONNEG>(v[u].z), i + 2);
        f(okey<NONNEG>(v[u].w), i + 3);
      }
    }
  }
  const int t = threadIdx.x, nt = n - sp.tail;
  if (t < sp.pre) f(okey<NONNEG>(__ldg(zm + t)), flat0 + (uint32_t)t);
  else if (t < sp.pre + nt) {
    const int i = sp.tail + (t - sp.pre);
    f(okey<NONNEG>(__ldg(zm + i)), flat0 + (uint32_t)i);
  }
}

// Calls f(order key, flat index) for the middle pairs of this warp's range (see
// warp_of), eight 16-byte loads in flight per lane.
template <typename F>
__device__ __forceinline__ void for_warp(const float *__restrict__ zm, uint32_t flat0, int n, F &&f) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Split sp = split_of(zm, n);
  const float4 *z4 = reinterpret_cast<const float4 *>(zm + sp.pre);
  const int per4 = (sp.n4 + NW - 1) / NW;
  const int b0 = min(sp.n4, warp * per4), b1 = min(sp.n4, b0 + per4);
  if (warp == 0 && lane < sp.pre) f(order_key(__ldg(zm + lane)), flat0 + (uint32_t)lane);
  for (int q0 = b0 + lane; q0 < b1; q0 += 8 * 32) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = q0 + 32 * u;
      v[u] = q < b1 ? __ldg(z4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = q0 + 32 * u;
      if (q < b1) {
        const uint32_t i = flat0 + (uint32_t)(sp.pre + 4 * q);
        f(order_key(v[u].x), i);
        f(order_key(v[u].y), i + 1);
        f(order_key(v[u].z), i + 2);
        f(order_key(v[u].w), i + 3);
      }
    }
  }
  if (warp == NW - 1 && lane < n - sp.tail)
    f(order_key(__ldg(zm + sp.tail + lane)), flat0 + (uint32_t)(sp.tail + lane));
}

// Bitmask of a head's kept middle pairs, laid out by the warp ranges of
// for_warp: warp w, round s (its vectors b0 + 256 s + [0, 256)) and lane l own
// one word whose nibble u holds the four pairs of vector b0 + 256 s + 32 u + l;
// two more words hold the leading and the trailing scalars.  nrw: rounds per
// warp range; a head takes bm_words(nrw) words.
__host__ __device__ __forceinline__ int bm_words(int nrw) { return NW * nrw * 32 + 2; }
// rounds for any head with n middle pairs (a head has at most n/4 vectors)
__host__ __device__ __forceinline__ int bm_rounds(int n) { return (((n >> 2) + NW - 1) / NW + 255) / 256; }
// Sets the bit of middle position i (shared-memory atomics: the word's other
// bits may be set at the same time).
__device__ __forceinline__ void bm_set(uint32_t *bm, int nrw, const Split &sp, int i) {
  if (i < sp.pre) {
    atomicOr(&bm[NW * nrw * 32], 1u << i);
  } else if (i >= sp.tail) {
    atomicOr(&bm[NW * nrw * 32 + 1], 1u << (i - sp.tail));
  } else {
    const int per4 = (sp.n4 + NW - 1) / NW;
    const int q = (i - sp.pre) >> 2, c = (i - sp.pre) & 3;
    const int w = q / per4, off = q - w * per4;
    atomicOr(&bm[(w * nrw + (off >> 8)) * 32 + (off & 31)], 1u << (4 * ((off >> 5) & 7) + c));
  }
}

// Step 3's stream over this warp's range (the ranges of for_warp, eight 16-byte
// loads in flight per lane): visit(order key, flat index) for every middle pair,
// returning whether the pair is kept for sure; with bm those answers go to the
// head's bitmask (every word of this warp's rounds is written).
template <bool NONNEG, typename V>
__device__ __forceinline__ void gather_stream(const float *__restrict__ zm, uint32_t flat0, int n,
                                              uint32_t *bm, int nrw, V &&visit) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Split sp = split_of(zm, n);
  const float4 *z4 = reinterpret_cast<const float4 *>(zm + sp.pre);
  const int per4 = (sp.n4 + NW - 1) / NW;
  const int b0 = min(sp.n4, warp * per4), b1 = min(sp.n4, b0 + per4);
  if (warp == 0) {
    bool k = false;
    if (lane < sp.pre) k = visit(okey<NONNEG>(__ldg(zm + lane)), flat0 + (uint32_t)lane);
    const unsigned m = __ballot_sync(0xFFFFFFFFu, k);
    if (bm && lane == 0) bm[NW * nrw * 32] = m;
  }
  const int nit = (b1 - b0 + 255) / 256;
  for (int r = 0; r < nit; ++r) {
    const int q0 = b0 + 256 * r + lane;
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = q0 + 32 * u;
      v[u] = q < b1 ? __ldg(z4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    uint32_t word = 0u;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = q0 + 32 * u;
      if (q < b1) {
        const uint32_t i = flat0 + (uint32_t)(sp.pre + 4 * q);
        uint32_t bits = visit(okey<NONNEG>(v[u].x), i) ? 1u : 0u;
        bits |= visit(okey<NONNEG>(v[u].y), i + 1) ? 2u : 0u;
        bits |= visit(okey<NONNEG>(v[u].z), i + 2) ? 4u : 0u;
        bits |= visit(okey<NONNEG>(v[u].w), i + 3) ? 8u : 0u;
        word |= bits << (4 * u);
      }
    }
    if (bm) bm[(warp * nrw + r) * 32 + lane] = word;
  }
  if (warp == NW - 1) {
    bool k = false;
    if (lane < n - sp.tail) k = visit(okey<NONNEG>(__ldg(zm + sp.tail + lane)), flat0 + (uint32_t)(sp.tail + lane));
    const unsigned m = __ballot_sync(0xFFFFFFFFu, k);
    if (bm && lane == 0) bm[NW * nrw * 32 + 1] = m;
  }
}

// Calls f(order key) for the pairs of every 16th vector of one head's middle
// range (a sample of about n/16 pairs); returns the sample's size.
template <typename F>
__device__ __forceinline__ int for_sample(const float *__restrict__ zm, int n, F &&f) {
  const Split sp = split_of(zm, n);
  const float4 *z4 = reinterpret_cast<const float4 *>(zm + sp.pre);
  const int ns4 = (sp.n4 + 15) / 16;
  for (int base = threadIdx.x; base < ns4; base += 4 * NT) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = base + u * NT;
      v[u] = j < ns4 ? __ldg(z4 + 16 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (base + u * NT < ns4) {
        f(order_key(v[u].x));
        f(order_key(v[u].y));
        f(order_key(v[u].z));
        f(order_key(v[u].w));
      }
  }
  return 4 * ns4;
}

// gs[g] = the counts of bins [64 g, 64 g + 64) of a kBins histogram (8 threads a
// group).  Every thread of the CTA must call; the caller synchronises after.
__device__ __forceinline__ void group_sums(const uint32_t *h, uint32_t *gs) {
  static_assert(kGroups * 8 == NT && kBins == kGroups * 64, "group layout");
  const int g = threadIdx.x >> 3, part = threadIdx.x & 7;
  uint32_t c = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) c += h[g * 64 + part * 8 + i];
  c += __shfl_xor_sync(0xFFFFFFFFu, c, 1);
  c += __shfl_xor_sync(0xFFFFFFFFu, c, 2);
  c += __shfl_xor_sync(0xFFFFFFFFu, c, 4);
  if (part == 0) gs[g] = c;
}

// Warp 0: in the sum over the cluster's ranks of the kBins histograms h (with
// their group sums gs, both at the same shared-memory offsets in every rank),
// taken from the top, the bin where the count first reaches `need`: sm.bin and
// sm.need (sm.bin = -1 when the counts never reach it).  Reads the 64 group
// sums and then one group's 64 bins of every rank.
__device__ void cluster_boundary(cg::cluster_group &cl, int CL, const uint32_t *h,
                                 const uint32_t *gs, uint32_t need, Smem &sm) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) sm.bin = -1;
  __syncwarp();
  uint32_t c0 = 0, c1 = 0;  // lane l: groups 63 - 2l and 62 - 2l
#pragma unroll
  for (int r = 0; r < kMaxCluster; ++r)
    if (r < CL) {
      const uint32_t *cc = cl.map_shared_rank(gs, r);
      c0 += cc[kGroups - 1 - 2 * lane];
      c1 += cc[kGroups - 2 - 2 * lane];
    }
  uint32_t incl = c0 + c1;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += y;
  }
  uint32_t above = incl - (c0 + c1);
  bool has = above < need && need <= incl;
  int G = 0;
  uint32_t aboveG = 0;
  if (has) {
    if (need <= above + c0) {
      G = kGroups - 1 - 2 * lane;
      aboveG = above;
    } else {
      G = kGroups - 2 - 2 * lane;
      aboveG = above + c0;
    }
  }
  const int src = (__ffs(__ballot_sync(0xFFFFFFFFu, has)) - 1) & 31;
  G = __shfl_sync(0xFFFFFFFFu, G, src);
  aboveG = __shfl_sync(0xFFFFFFFFu, aboveG, src);
  uint32_t f0 = 0, f1 = 0;  // lane l: bins 64G + 63 - 2l and 64G + 62 - 2l
  const int e0 = G * 64 + 63 - 2 * lane;
#pragma unroll
  for (int r = 0; r < kMaxCluster; ++r)
    if (r < CL) {
      const uint32_t *cc = cl.map_shared_rank(h, r);
      f0 += cc[e0];
      f1 += cc[e0 - 1];
    }
  incl = f0 + f1;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += y;
  }
  above = aboveG + incl - (f0 + f1);
  has = above < need && need <= aboveG + incl;
  if (has) {
    const bool first = need <= above + f0;
    sm.bin = first ? e0 : e0 - 1;
    sm.need = (int)(need - (first ? above : above + f0));
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

// Exact threshold inside one bucket (the keys' top 20 bits fixed to those of
// `prefix`): the key with exactly `need` of the visited bucket keys at or above
// it.  8-bit digits below the bucket's bits, stopping once a digit's bucket is
// taken whole; keys are unique, so the last digit always settles it.  visit(f)
// calls f(key) for every candidate this thread owns (keys outside the bucket
// are ignored).  Every thread of the CTA must call.
template <typename Visit>
__device__ uint64_t select_in_bucket(Smem &sm, uint64_t prefix, int need, Visit visit) {
  const int warp = threadIdx.x >> 5;
  uint64_t hmask = ~0ull << kSubShift;
  for (int shift = kSubShift - 8;; shift -= 8) {
    const int sh = max(shift, 0);
    const uint32_t dmask = shift >= 0 ? 255u : (255u >> -shift);
    for (int d = threadIdx.x; d < 256; d += NT) sm.h256[d] = 0u;
    __syncthreads();
    visit([&](uint64_t key) {
      if ((key & hmask) == prefix) atomicAdd(&sm.h256[(uint32_t)(key >> sh) & dmask], 1u);
    });
    __syncthreads();
    if (warp == 0) digit_boundary(sm.h256, need, prefix, sh, sm.rx);
    __syncthreads();
    prefix = sm.rx.sh_prefix;
    need = sm.rx.sh_need;
    hmask |= (uint64_t)dmask << sh;
    const int done = sm.rx.sh_done;
    __syncthreads();  // h256 and sh_* are rewritten by the next digit
    if (done || sh == 0) break;
  }
  return prefix;
}

__global__ __launch_bounds__(NT, 2) void select_budget_kernel(
    const float *__restrict__ z, int H, int T, int budget, int floor_k, int R, int S,
    int32_t *__restrict__ idx_out, int32_t *__restrict__ off_out) {
  __shared__ Smem sm;
  extern __shared__ __align__(16) unsigned char dyn_raw[];
  Dyn &dy = *reinterpret_cast<Dyn *>(dyn_raw);
  uint32_t *const bm_all = reinterpret_cast<uint32_t *>(dyn_raw + sizeof(Dyn));  // [kBmWords]
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
  // head and middle position of a pair key
  auto head_of = [&](uint64_t key) { return (int)((0xFFFFFFFFu - (uint32_t)key) / (uint32_t)T); };
  auto pos_of = [&](uint64_t key) {
    const uint32_t flat = 0xFFFFFFFFu - (uint32_t)key;
    return (int)(flat % (uint32_t)T) - S;
  };

  for (int e = threadIdx.x; e < kBins; e += NT) dy.h.comp[e] = 0u;

  // 0. With one head per CTA (H <= 8), the bins of theta_h and of tau are
  //    predicted from a sample of every 16th vector, so that the first stream
  //    can also take the second digits of three bins around each prediction
  //    and the digit stream is needed only where a prediction missed.  The
  //    sample's competition counts go to the bitmask area, which is not written
  //    before step 3, so the ranks can read them without another barrier.
  const bool pred = H <= kMaxCluster;
  int w1 = -8, wt = -8;  // first bin of each three-bin window (-8: none)
  if (pred) {
    const int h = rank;
    uint32_t *const scomp = bm_all;           // [kBins] the sample's competition counts
    uint32_t *const sgrp = bm_all + kBins;    // [kGroups] their group sums
    for (int e = threadIdx.x; e < kBins; e += NT) dy.h.hist[e] = 0u;
    for (int e = threadIdx.x; e < 6 * 256; e += NT) (&sm.wsub[0][0])[e] = 0u;
    __syncthreads();
    const int ns = for_sample(zmid(h), n, [&](uint32_t ok) { atomicAdd(&dy.h.hist[ok >> kBinShift32], 1u); });
    __syncthreads();
    int b1e = kBins, need1e = 0;
    if (nf > 0 && ns > 0) {
      const int nfs = (int)min((long long)ns, max(1LL, ((long long)nf * ns + n / 2) / n));
      find_boundary(dy.h.hist, nfs, sm);
      b1e = sm.bin;
      need1e = sm.need;
      w1 = b1e - 1;
    }
    for (int e = threadIdx.x; e < kBins; e += NT)
      scomp[e] = e < b1e ? dy.h.hist[e] : e == b1e ? dy.h.hist[e] - (uint32_t)need1e : 0u;
    __syncthreads();
    group_sums(scomp, sgrp);
    cl.sync();  // every CTA of the cluster is running, and every sample's counts are complete
    if (extra > 0 && ns > 0) {
      const uint32_t es = (uint32_t)max(1LL, ((long long)extra * ns + n / 2) / n);
      if (warp == 0) cluster_boundary(cl, CL, scomp, sgrp, es, sm);
      __syncthreads();
      if (sm.bin >= 0) wt = sm.bin - 1;
    }
  } else {
    cl.sync();  // every CTA of the cluster is running before any remote access
  }
  // the window slot of bin b (0..2 theta's, 3..5 tau's), -1 outside both
  auto wslot = [&](int b) {
    const uint32_t d1 = (uint32_t)(b - w1), dt = (uint32_t)(b - wt);
    return d1 < 3u ? (int)d1 : dt < 3u ? 3 + (int)dt : -1;
  };

  // 1. per owned head, the 12-bit histogram: theta_h's bin, and from the counts
  //    alone this head's share of the competition's 12-bit histogram (the bins
  //    below theta_h's whole, theta_h's bin less the need1 pairs at or above it)
  for (int h = rank, j = 0; h < H; h += CL, ++j) {
    for (int e = threadIdx.x; e < kBins; e += NT) dy.h.hist[e] = 0u;
    __syncthreads();
    if (pred) {
      for_head(zmid(h), flat0(h), n, [&](uint32_t ok, uint32_t) {
        const int b = (int)(ok >> kBinShift32);
        atomicAdd(&dy.h.hist[b], 1u);
        const int sl = wslot(b);
        if (sl >= 0) atomicAdd(&sm.wsub[sl][(ok >> kSubShift32) & 255u], 1u);
      });
    } else {
      for_head(zmid(h), flat0(h), n, [&](uint32_t ok, uint32_t) { atomicAdd(&dy.h.hist[ok >> kBinShift32], 1u); });
    }
    __syncthreads();
    {
      // negative scores have keys below 2^31: bins [0, kBins / 2)
      uint32_t negs = 0u;
      for (int e = threadIdx.x; e < kBins / 2; e += NT) negs |= dy.h.hist[e];
      const int nonneg = !__syncthreads_or(negs != 0u);
      if (threadIdx.x == 0) sm.nonneg[j] = nonneg;
    }
    int b1 = kBins, need1 = 0;  // b1 = kBins: no floor, every pair below theta_h
    if (nf > 0) {
      find_boundary(dy.h.hist, nf, sm);
      b1 = sm.bin;
      need1 = sm.need;
    }
    if (threadIdx.x == 0) {
      sm.b1[j] = b1;
      sm.need1[j] = need1;
      sm.p20h[j] = ~0u;  // no bucket to gather (set below when there is one)
      sm.big[j] = 0;
    }
    for (int e = threadIdx.x; e < kBins; e += NT)
      if (e < b1) dy.h.comp[e] += dy.h.hist[e];
      else if (e == b1) dy.h.comp[e] += dy.h.hist[e] - (uint32_t)need1;
    __syncthreads();  // hist serves the next head
  }
  group_sums(dy.h.comp, sm.ccoarse);  // this CTA's competition counts per group
  cl.sync();  // every competition histogram complete

  // 2. tau's bin from the cluster's sum; one stream per owned head takes the
  //    second digits of theta_h's bin and, where that bin lies above tau's,
  //    of tau's bin (all of whose pairs are then below theta_h)
  int bt = -1, needt1 = 0;
  if (extra > 0) {
    // from the cluster's sums taken from the top: the group of bins where the
    // count reaches `extra`, then the bin inside it (4 KB of remote reads
    // instead of every rank's 4096 bins)
    if (warp == 0) cluster_boundary(cl, CL, dy.h.comp, sm.ccoarse, (uint32_t)extra, sm);
    __syncthreads();
    bt = sm.bin;
    needt1 = sm.need;
  }
  uint32_t *const h8c = sm.h8 + 256;
  for (int d = threadIdx.x; d < 256; d += NT) h8c[d] = 0u;
  for (int h = rank, j = 0; h < H; h += CL, ++j) {
    const int b1 = sm.b1[j];
    const int bc = bt < b1 ? bt : -2;  // tau's bin when below theta_h's (-2: no bin)
    if (b1 == kBins && bc < 0) continue;  // uniform over the CTA: nothing to count
    // digits the first stream took (predicted bins); the stream takes the rest
    const int s1 = pred && b1 < kBins ? wslot(b1) : -1;
    const int sc = pred && bc >= 0 ? wslot(bc) : -1;
    const int b1s = b1 < kBins && s1 < 0 ? b1 : -1;
    const int bcs = bc >= 0 && sc < 0 ? bc : -2;
    for (int d = threadIdx.x; d < 256; d += NT) sm.h8[d] = s1 >= 0 ? sm.wsub[s1][d] : 0u;
    if (sc >= 0)
      for (int d = threadIdx.x; d < 256; d += NT) h8c[d] += sm.wsub[sc][d];
    __syncthreads();
    if (b1s >= 0 || bcs >= 0) {
      auto digits = [&](uint32_t ok, uint32_t) {
        const int b = (int)(ok >> kBinShift32);
        const bool in1 = b == b1s;
        if (in1 || b == bcs) atomicAdd(&sm.h8[(in1 ? 0u : 256u) + ((ok >> kSubShift32) & 255u)], 1u);
      };
      if (sm.nonneg[j]) for_head<true>(zmid(h), flat0(h), n, digits);
      else for_head<false>(zmid(h), flat0(h), n, digits);
      __syncthreads();
    }
    if (b1 < kBins) {
      if (warp == 0) digit_boundary(sm.h8, sm.need1[j], (uint64_t)b1 << kBinShift, kSubShift, sm.rx);
      __syncthreads();
      const uint64_t pb = sm.rx.sh_prefix;  // theta_h's bucket: its top 20 bits, zeros below
      const int need2 = sm.rx.sh_need;
      const int d2 = (int)((pb >> kSubShift) & 255u);
      if (threadIdx.x == 0) {
        sm.p20h[j] = (uint32_t)(pb >> kSubShift);
        sm.need2[j] = need2;
        sm.big[j] = sm.h8[d2] > (uint32_t)kListCap;
      }
      // tau's bin is theta_h's: the competition takes the bin's pairs below theta_h
      if (b1 == bt)
        for (int d = threadIdx.x; d < 256; d += NT)
          h8c[d] += d < d2 ? sm.h8[d] : d == d2 ? sm.h8[d] - (uint32_t)need2 : 0u;
    }
    __syncthreads();  // h8 and the sh_* fields serve the next head
  }
  cl.sync();  // every second-digit histogram complete

  uint64_t pt = 0;
  uint32_t p20t = ~0u;  // tau's bucket (~0u: no competition)
  int needt2 = 0;
  if (extra > 0) {
    for (int d = threadIdx.x; d < 256; d += NT) {
      uint32_t g = 0;
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < CL) g += cl.map_shared_rank(h8c, r)[d];
      sm.g8[d] = g;
    }
    __syncthreads();
    if (warp == 0) digit_boundary(sm.g8, needt1, (uint64_t)bt << kBinShift, kSubShift, sm.rx);
    __syncthreads();
    pt = sm.rx.sh_prefix;
    needt2 = sm.rx.sh_need;
    p20t = (uint32_t)(pt >> kSubShift);
    __syncthreads();  // the sh_* fields are rewritten by the selects below
  }

  // 3. per owned head, one stream gathers theta_h's bucket and tau's (every pair
  //    of it, kept by its floor or not) and counts per warp range the pairs above
  //    each; theta_h follows from its bucket's pairs at once
  const int nrw = bm_rounds(n), bm_stride = bm_words(nrw);
  if (threadIdx.x == 0) sm.list_n = 0;
  for (int h = rank, j = 0; h < H; h += CL, ++j) {
    const float *zm = zmid(h);
    const uint32_t f0 = flat0(h);
    const Split sp = split_of(zm, n);
    const int per4 = max(1, (sp.n4 + NW - 1) / NW);
    const int big = sm.big[j];
    const uint32_t ph = big ? ~0u : sm.p20h[j];  // ~0u: matches no pair
    // The head's threshold min(theta_h, tau) lies in the lower of the two
    // buckets: the pairs of higher buckets are kept for sure (the bitmask), those
    // of that bucket are taken from its list once the thresholds are known.
    const uint32_t pl = min(ph, p20t);
    const bool use_bm = !big && (ph != ~0u || p20t != ~0u) && (j + 1) * bm_stride <= kBmWords;
    uint32_t *const bmh = use_bm ? bm_all + j * bm_stride : nullptr;
    if (threadIdx.x == 0) {
      sm.tl_n = 0;
      sm.bmok[j] = use_bm;
    }
    __syncthreads();
    int c1 = 0, c2 = 0;
    if (ph != ~0u || p20t != ~0u) {
      auto visit = [&](uint32_t ok, uint32_t fl) {
        const uint32_t pk = ok >> kSubShift32;
        c1 += pk > ph;
        c2 += pk > p20t;
        if (pk == ph || pk == p20t) {  // rare
          if (pk == ph) dy.l.tlist[atomicAdd(&sm.tl_n, 1)] = pair_key_u(ok, fl);  // <= kListCap pairs
          if (pk == p20t) {
            const int slot = atomicAdd(&sm.list_n, 1);
            if (slot < kListCap) dy.l.clist[slot] = pair_key_u(ok, fl);
          }
        }
        return pk > pl;
      };
      if (sm.nonneg[j]) gather_stream<true>(zm, f0, n, bmh, nrw, visit);
      else gather_stream<false>(zm, f0, n, bmh, nrw, visit);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        c1 += __shfl_xor_sync(0xFFFFFFFFu, c1, off);
        c2 += __shfl_xor_sync(0xFFFFFFFFu, c2, off);
      }
    }
    if (lane == 0) {
      sm.wth[j][warp] = c1;
      sm.wtau[j][warp] = c2;
    }
    __syncthreads();
    uint64_t th = kNone;
    int ok = 1;  // wth[j] holds the per-warp counts of pairs >= th
    if (sm.b1[j] < kBins) {
      if (!big) {
        const int ln = sm.tl_n;
        const uint64_t pb = (uint64_t)ph << kSubShift;
        th = select_in_bucket(sm, pb, sm.need2[j], [&](auto &&f) {
          for (int i = threadIdx.x; i < ln; i += NT) f(dy.l.tlist[i]);
        });
        th = max(th, pb);  // the select stops at the first digit that settles the bucket
        // theta_h's bucket below tau's: the head's threshold is theta_h
        const bool mark = use_bm && ph < p20t;
        for (int i = threadIdx.x; i < ln; i += NT) {
          const uint64_t key = dy.l.tlist[i];
          if (key >= th) {
            atomicAdd(&sm.wth[j][warp_of(pos_of(key), sp, per4)], 1);
            if (mark) bm_set(bmh, nrw, sp, pos_of(key));
          }
        }
      } else {
        th = radix_select_ge<NT, false>(sm.rx, nf, [&](auto &&f) {
          for_head(zm, f0, n, [&](uint32_t ok, uint32_t fl) { f(pair_key_u(ok, fl)); });
        });
        ok = 0;
      }
    }
    if (threadIdx.x < CL) cl.map_shared_rank(sm.theta, threadIdx.x)[h] = th;
    if (threadIdx.x == 0) sm.thok[j] = ok;
    __syncthreads();  // the theta list serves the next head
  }

  // tau from the cluster's gathered pairs below their head's theta
  uint64_t tau = kNone;
  int tau_ok = 0;  // wtau and the list hold tau's counts
  if (threadIdx.x < CL) {
    cl.map_shared_rank(sm.lnr, threadIdx.x)[rank] = min(sm.list_n, kListCap);
    cl.map_shared_rank(sm.ovr, threadIdx.x)[rank] = sm.list_n > kListCap;
  }
  cl.sync();  // every theta and every bucket list complete
  if (extra > 0) {
    int ovf = 0, ltot = 0;
    for (int r = 0; r < CL; ++r) {
      ovf |= sm.ovr[r];
      ltot += sm.lnr[r];
    }
    if (!ovf) {
      // the lists as one sequence, rank by rank, read in place
      auto list_at = [&](int q) {
        int r = 0;
        while (q >= sm.lnr[r]) q -= sm.lnr[r++];
        return cl.map_shared_rank(dy.l.clist, r)[q];
      };
      tau = select_in_bucket(sm, pt, needt2, [&](auto &&f) {
        for (int q = threadIdx.x; q < ltot; q += NT) {
          const uint64_t key = list_at(q);
          if (key < sm.theta[head_of(key)]) f(key);
        }
      });
      tau = max(tau, pt);  // as for the floor thresholds
      tau_ok = 1;
    } else {
      tau = radix_select_ge<NT, true>(sm.rx, (int)extra, [&](auto &&f) {
        for (int h = rank; h < H; h += CL) {
          const uint64_t th = sm.theta[h];
          for_head(zmid(h), flat0(h), n, [&](uint32_t ok, uint32_t fl) {
            if (!key_ge(ok, fl, th)) f(pair_key_u(ok, fl));
          });
        }
      });
    }
  }

  // kept middle pairs per owned head and warp range; counts to every CTA
  for (int h = rank, j = 0; h < H; h += CL, ++j) {
    const uint64_t th = sm.theta[h];
    const uint64_t lam = min(th, tau);
    const float *zm = zmid(h);
    const uint32_t f0 = flat0(h);
    const Split sp = split_of(zm, n);
    const int per4 = max(1, (sp.n4 + NW - 1) / NW);
    if (lam == th && sm.thok[j]) {
      if (threadIdx.x < NW) sm.wcnt[j][threadIdx.x] = sm.wth[j][threadIdx.x];
      __syncthreads();
    } else if (lam == tau && tau_ok) {
      if (threadIdx.x < NW) sm.wcnt[j][threadIdx.x] = sm.wtau[j][threadIdx.x];
      __syncthreads();
      const int ln = min(sm.list_n, kListCap);
      for (int i = threadIdx.x; i < ln; i += NT) {
        const uint64_t key = dy.l.clist[i];
        if (head_of(key) == h && key >= lam) atomicAdd(&sm.wcnt[j][warp_of(pos_of(key), sp, per4)], 1);
      }
    } else {
      // a counting stream over the warp ranges
      int c = 0;
      for_warp(zm, f0, n, [&](uint32_t ok, uint32_t fl) { c += key_ge(ok, fl, lam); });
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
      if (lane == 0) sm.wcnt[j][warp] = c;
    }
    // tau's bucket at or below theta_h's: the head's kept pairs of that bucket
    // are marked from the competition's list (no list, no bitmask)
    bool bm_use = sm.bmok[j];
    if (bm_use && p20t <= (sm.big[j] ? ~0u : sm.p20h[j])) {
      if (tau_ok) {
        const int ln = min(sm.list_n, kListCap);
        for (int i = threadIdx.x; i < ln; i += NT) {
          const uint64_t key = dy.l.clist[i];
          if (head_of(key) == h && key >= lam) bm_set(bm_all + j * bm_stride, nrw, sp, pos_of(key));
        }
      } else {
        bm_use = false;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) sm.bmok[j] = bm_use;
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
    const uint32_t lam_hi = (uint32_t)(lam >> 32);
    // L0: the threshold's low word is zero, so the order key alone decides
    auto emit = [&](auto low0) {
      constexpr bool L0 = decltype(low0)::value;
      auto ge = [&](uint32_t ok, uint32_t fl) { return L0 ? ok >= lam_hi : key_ge(ok, fl, lam); };
      if (warp == 0) {
        const bool keep = lane < sp.pre && ge(order_key(__ldg(zm + lane)), f0 + (uint32_t)lane);
        const unsigned m = __ballot_sync(0xFFFFFFFFu, keep);
        const int slot = run + __popc(m & below);
        if (keep && slot < kept_mid) mid[slot] = S + lane;
        run += __popc(m);
      }
      for (int q00 = b0; q00 < b1; q00 += 4 * 32) {  // four vectors a lane in flight
        float4 vv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int q = q00 + 32 * u + lane;
          vv[u] = q < b1 ? __ldg(z4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // keep bits of each vector, and their counts packed one byte per vector
        // (at most 4 x 32 = 128 a byte, so one scan serves all four)
        uint32_t kb[4], packed = 0u;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int q = q00 + 32 * u + lane;
          uint32_t bits = 0u;
          if (q < b1) {
            const float4 v = vv[u];
            const uint32_t fi = f0 + (uint32_t)(sp.pre + 4 * q);
            bits = (uint32_t)ge(order_key(v.x), fi) | (uint32_t)ge(order_key(v.y), fi + 1) << 1 |
                   (uint32_t)ge(order_key(v.z), fi + 2) << 2 | (uint32_t)ge(order_key(v.w), fi + 3) << 3;
          }
          kb[u] = bits;
          packed |= (uint32_t)__popc(bits) << (8 * u);
        }
        uint32_t incl = packed;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
          if (lane >= off) incl += y;
        }
        const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
        const uint32_t excl = incl - packed;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          int slot = run + (int)((excl >> (8 * u)) & 255u);
          const int i = sp.pre + 4 * (q00 + 32 * u + lane);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if ((kb[u] >> c) & 1u) {
              if (slot < kept_mid) mid[slot] = S + i + c;
              ++slot;
            }
          run += (int)((tot >> (8 * u)) & 255u);
        }
      }
      if (warp == NW - 1) {
        const int i = sp.tail + lane;
        const bool keep = i < n && ge(order_key(__ldg(zm + i)), f0 + (uint32_t)i);
        const unsigned m = __ballot_sync(0xFFFFFFFFu, keep);
        const int slot = run + __popc(m & below);
        if (keep && slot < kept_mid) mid[slot] = S + i;
      }
    };
    if (sm.bmok[j]) {
      // from the head's bitmask: nibble u of lane l's word of round r holds
      // vector b0 + 256 r + 32 u + l; the eight vectors' counts packed one byte
      // each (at most 128) share one scan
      const uint32_t *bmh = bm_all + j * bm_stride;
      if (warp == 0) {
        const unsigned m = bmh[NW * nrw * 32];
        const int slot = run + __popc(m & below);
        if (((m >> lane) & 1u) && slot < kept_mid) mid[slot] = S + lane;
        run += __popc(m);
      }
      const int nit = (b1 - b0 + 255) / 256;
      for (int r = 0; r < nit; ++r) {
        const uint32_t word = bmh[(warp * nrw + r) * 32 + lane];
        uint64_t packed = 0u;
#pragma unroll
        for (int u = 0; u < 8; ++u) packed |= (uint64_t)__popc((word >> (4 * u)) & 15u) << (8 * u);
        uint64_t incl = packed;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
          if (lane >= off) incl += y;
        }
        const uint64_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
        const uint64_t excl = incl - packed;
        // the round's kept pairs before vector u, as 16-bit fields (at most 1024)
        uint64_t cum_lo = 0u, cum_hi = 0u;
        uint32_t acc = 0u;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (u < 4) cum_lo |= (uint64_t)acc << (16 * u);
          else cum_hi |= (uint64_t)acc << (16 * (u - 4));
          acc += (uint32_t)(tot >> (8 * u)) & 255u;
        }
        // only the set bits (a head keeps a few percent of its middle pairs)
        for (uint32_t w = word; w; w &= w - 1u) {
          const int b = __ffs(w) - 1, u = b >> 2, c = b & 3;
          const uint64_t cum = u < 4 ? cum_lo : cum_hi;
          const int slot = run + (int)((cum >> (16 * (u & 3))) & 0xFFFFu) +
                           (int)((excl >> (8 * u)) & 255u) + __popc((word >> (4 * u)) & ((1u << c) - 1u));
          if (slot < kept_mid) mid[slot] = S + sp.pre + 4 * (b0 + 256 * r + 32 * u + lane) + c;
        }
        run += (int)acc;
      }
      if (warp == NW - 1) {
        const unsigned m = bmh[NW * nrw * 32 + 1];
        const int slot = run + __popc(m & below);
        if (((m >> lane) & 1u) && slot < kept_mid) mid[slot] = S + sp.tail + lane;
      }
    } else if ((uint32_t)lam == 0u) {
      emit(std::true_type{});
    } else {
      emit(std::false_type{});
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
  const size_t dyn = sizeof(Dyn) + sizeof(uint32_t) * kBmWords;
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = st;
  if (ensure_smem((const void *)select_budget_kernel, dyn))
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
