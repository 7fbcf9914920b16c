// select_topk.cu -- budgeted per-head Top-K with a protected recent window.
//
// H2O page, 双缓冲 and 为什么要按头独立驱逐: every head keeps the last R
// positions and the k - R best of [0, T - R) in the order (z descending,
// position ascending); the kept positions are written in ascending order.
// With S sinks (KV-cache survey blog §4.1-4.2) the first S positions are kept
// too and the heavy part is the k - R - S best of [S, T - R).
//
// Resident kernel (every head with at most 8 x 49152 candidates): one
// thread-block cluster of CL CTAs per head; CTA c holds its contiguous slice of
// the head's candidates in shared memory as order-preserving keys, so z is read
// from HBM exactly once.  Each candidate's 64-bit key (z's key, ~position) is
// unique and orders exactly as (z descending, position ascending); a radix
// select over the slices (histograms summed through distributed shared memory)
// finds the threshold with exactly k - R - S keys at or above it.  Per-warp
// counts over contiguous ranges, an exclusive sum over the cluster's CTAs, and
// warp ballots emit the kept positions already ascending.
//
// Streaming kernel (longer heads): one 1024-thread block per head re-reads z
// (from L2) once per radix pass:
//   1. exact radix select (4 passes of 8 bits over order-preserving uint32
//      keys, per-warp shared-memory histograms) finds the (k-R)-th largest key u*
//      and how many of the keys equal to u* must be taken;
//   2. one ordered pass keeps every key > u* and the first `need` keys == u*
//      (block-wide scans give each kept position its output slot), so the
//      positions come out ascending without a sort;
//   3. the recent window is appended.
// Integer work only after the key transform: the same z always gives the same idx.
#include <cooperative_groups.h>

#include "kvc_internal.cuh"
#include "refine_common.cuh"
#include "select_common.cuh"

namespace cg = cooperative_groups;

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

constexpr int NTC = 512;            // threads of the resident kernel
constexpr int NWC = NTC / 32;
constexpr int kSliceSmall = 16384;  // keys per CTA with two CTAs per SM
constexpr int kSliceMax = 49152;    // keys per CTA at most (192 KB)
constexpr int kMaxCl = 8;
// Radix histogram copies of the resident kernel (each shared by four warps): the
// smaller scratch lets three CTAs share an SM when their registers allow it.
constexpr int kHistCopies = 4;

struct ResidentSmem {
  RadixScratch<NTC, kHistCopies> rx;
  int wcnt[NWC];
  int cnt[kMaxCl];
};

// HubKV refinement folded into the selection's load (hubkv_select_topk): the
// kernel reads the base scores s and forms each candidate's z itself.
struct RefineArgs {
  const float *beta;  // [heads] head weights
  float *z_out;       // [heads][T], may be null
  float gamma, r2;
  int half;           // pool_width / 2
};

// MODE 0: z is given.  MODE 1 / 2: z is formed from s with the local-hub /
// average-pool discount (refine_common.cuh).
template <int MODE>
__global__ __launch_bounds__(NTC) void select_topk_resident_kernel(
    const float *__restrict__ z, int T, int k, int R, int S, int len,
    int32_t *__restrict__ idx_out, RefineArgs ra) {
  extern __shared__ __align__(16) unsigned char slice_raw[];
  __shared__ ResidentSmem sm;
  cg::cluster_group cl = cg::this_cluster();
  const int CL = (int)cl.num_blocks(), rank = (int)cl.block_rank();
  const long head = blockIdx.x / CL;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = T - R - S, nh = k - R - S;
  int32_t *out = idx_out + head * (long)k;
  const int lo = min(n, rank * len), hi = min(n, lo + len), m = hi - lo;
  const int half = MODE == 0 ? 0 : ra.half;
  const float *row = z + head * (long)T;  // z, or the base scores s (MODE 1 / 2)
  for (int e = threadIdx.x; e < kHistCopies * 256; e += NTC) (&sm.rx.hist[0][0])[e] = 0u;

  // The slice with a halo of `half` on each side (-inf past the prompt's ends):
  // tile[t] = row[p0 + t].  The tile starts `toff` floats into the buffer so
  // that it has the global addresses' 16-byte phase: the aligned middle moves
  // as 16-byte vectors, all in flight at once, the ragged ends as scalars.
  // The keys then replace the tile in place (key i at or left of tile[i]).
  const int p0 = S + lo - half, nt = m + 2 * half;
  const int rmis = (int)((reinterpret_cast<uintptr_t>(row) >> 2) & 3);
  const int toff = (((rmis + p0) % 4) + 4) % 4;
  float *tile = reinterpret_cast<float *>(slice_raw) + toff;
  uint32_t *keys = reinterpret_cast<uint32_t *>(slice_raw);
  {
    const int c0 = max(p0, 0), c1 = min(p0 + nt, T);
    const int a0 = min(c1, c0 + (4 - (rmis + c0) % 4) % 4);  // first 16-byte aligned index
    const int e0 = max(a0, c1 - (rmis + c1) % 4);            // end of the aligned run
    const int n4 = (e0 - a0) >> 2;
    const float4 *g4 = reinterpret_cast<const float4 *>(row + a0);
    float4 *t4 = reinterpret_cast<float4 *>(tile + (a0 - p0));
    for (int base = threadIdx.x; base < n4; base += 8 * NTC) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = base + u * NTC;
        v[u] = j < n4 ? __ldg(g4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = base + u * NTC;
        if (j < n4) t4[j] = v[u];
      }
    }
    const int front = a0 - p0, back = p0 + nt - e0;  // tile entries before a0, from e0 on
    for (int t = threadIdx.x; t < front + back; t += NTC) {
      const int tt = t < front ? t : (e0 - p0) + (t - front);
      const int p = p0 + tt;
      tile[tt] = (p >= 0 && p < T) ? __ldg(row + p) : -INFINITY;
    }
  }

  // z and the order keys, in batches of 8 x NTC candidates: every z of a batch
  // is formed before any of its keys lands (later batches read only further
  // right).  The first radix digit (the top byte) is counted here.
  const float beta = MODE == 0 ? 0.f : ra.beta[head];
  float *zo = (MODE != 0 && ra.z_out) ? ra.z_out + head * (long)T : nullptr;
  auto put = [&](int i, float zi) {
    const uint32_t kk = order_key(zi);
    keys[i] = kk;
    atomicAdd(&sm.rx.hist[warp & (kHistCopies - 1)][kk >> 24], 1u);
    if (zo) zo[S + lo + i] = zi;
  };
  if (MODE == 1 && half == 2) {
    // local hubs over a window of 5, four consecutive candidates a thread: the
    // 8 scores around them give the four window maxima from shared pair maxima
    // (the same values as hub_gate: a maximum does not depend on its order)
    const float g = ra.gamma, r2 = ra.r2;
    for (int base0 = 0; base0 < m; base0 += 8 * NTC) {
      __syncthreads();
      float v[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = base0 + 4 * (h * NTC + (int)threadIdx.x);
        if (c < m) {
          float w[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) w[q] = tile[c + q];  // s of candidates c-2 .. c+5
          const float m01 = fmaxf(w[0], w[1]), m23 = fmaxf(w[2], w[3]), m45 = fmaxf(w[4], w[5]),
                      m67 = fmaxf(w[6], w[7]);
          const float M[4] = {fmaxf(fmaxf(m01, m23), w[4]), fmaxf(fmaxf(w[1], m23), m45),
                              fmaxf(fmaxf(m23, m45), w[6]), fmaxf(fmaxf(w[3], m45), m67)};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float si = w[q + 2];
            const float qi = (si == M[q]) ? si : g * si;
            v[h][q] = fmaf(r2, fmaf(beta, qi, -si), si);
          }
        }
      }
      __syncthreads();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = base0 + 4 * (h * NTC + (int)threadIdx.x);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (c + q < m) put(c + q, v[h][q]);
      }
    }
  } else {
    for (int base0 = 0; base0 < m; base0 += 8 * NTC) {
      __syncthreads();
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base0 + threadIdx.x + u * NTC;
        v[u] = 0.f;
        if (i < m) {
          if constexpr (MODE == 0)
            v[u] = tile[i];
          else
            v[u] = hub_gate<MODE == 2>(tile + i + half, half, S + lo + i, T, ra.gamma, ra.r2, beta);
        }
      }
      __syncthreads();
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base0 + threadIdx.x + u * NTC;
        if (i < m) put(i, v[u]);
      }
    }
  }
  if (zo && rank == 0) {
    // z of the always-kept positions (sinks and recent window) for the caller,
    // windows read from global memory
    for (int e = threadIdx.x; e < S + R; e += NTC) {
      const int p = e < S ? e : T - R + (e - S);
      float win[2 * 64 + 1];
      for (int o = -half; o <= half; ++o)
        win[o + half] = (p + o >= 0 && p + o < T) ? __ldg(row + p + o) : -INFINITY;
      zo[p] = hub_gate<MODE == 2>(win + half, half, p, T, ra.gamma, ra.r2, beta);
    }
  }
  cl.sync();  // slices loaded, and every CTA of the cluster is running

  const uint64_t thr = radix_select_ge<NTC, true>(
      sm.rx, nh,
      [&](auto &&f) {
        for (int i = threadIdx.x; i < m; i += NTC) f(pair_key_u(keys[i], (uint32_t)(lo + i)));
      },
      [&](auto &&f) {
        const int m4 = m >> 2;  // four keys per 16-byte load
        const uint4 *k4 = reinterpret_cast<const uint4 *>(keys);
        for (int i = threadIdx.x; i < m4; i += NTC) {
          const uint4 q = k4[i];
          f(q.x);
          f(q.y);
          f(q.z);
          f(q.w);
        }
        for (int i = 4 * m4 + threadIdx.x; i < m; i += NTC) f(keys[i]);
      },
      true);
  // a threshold with a zero low word is decided by the order keys alone
  const bool thr32 = (uint32_t)thr == 0u;
  const uint32_t thr_hi = (uint32_t)(thr >> 32);
  auto kept = [&](int i) {
    return thr32 ? keys[i] >= thr_hi : pair_key_u(keys[i], (uint32_t)(lo + i)) >= thr;
  };

  // kept candidates per warp range, per CTA, then the CTA's output offset
  const int per = ((m + NWC - 1) / NWC + 31) & ~31;
  const int wlo = min(m, warp * per), whi = min(m, wlo + per);
  int c = 0;
  for (int i = wlo + lane; i < whi; i += 32) c += kept(i);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
  if (lane == 0) sm.wcnt[warp] = c;
  __syncthreads();
  if (threadIdx.x < CL) {
    int tot = 0;
    for (int w = 0; w < NWC; ++w) tot += sm.wcnt[w];
    cl.map_shared_rank(&sm.cnt[0], threadIdx.x)[rank] = tot;
  }
  cl.sync();  // the last remote access is above
  int run = 0;
  for (int r = 0; r < rank; ++r) run += sm.cnt[r];
  for (int w = 0; w < warp; ++w) run += sm.wcnt[w];
  for (int i0 = wlo; i0 < whi; i0 += 32) {
    const int i = i0 + lane;
    const bool keep = i < whi && kept(i);
    const unsigned msk = __ballot_sync(0xFFFFFFFFu, keep);
    const int slot = run + __popc(msk & ((1u << lane) - 1u));
    if (keep && slot < nh) out[S + slot] = S + lo + i;
    run += __popc(msk);
  }
  if (rank == 0) {
    for (int mm = threadIdx.x; mm < S; mm += NTC) out[mm] = mm;
    for (int mm = threadIdx.x; mm < R; mm += NTC) out[S + nh + mm] = S + n + mm;
  }
}

}  // namespace

namespace {

// Cluster geometry of the resident kernel for n candidates with nh heavy slots:
// CTAs per head and candidates per CTA (len 0: not resident).
void resident_plan(int n, int nh, int *CL, int *len) {
  *CL = 0;
  *len = 0;
  if (nh < n) {
    *CL = (n + kSliceSmall - 1) / kSliceSmall;
    if (*CL > kMaxCl && n <= kMaxCl * kSliceMax) *CL = kMaxCl;
    if (*CL <= kMaxCl) *len = (n + *CL - 1) / *CL;
  }
}

template <int MODE>
int launch_resident(const float *z, long heads, int T, int k, int recent, int sink, int CL, int len,
                    int halo, int32_t *idx, const RefineArgs &ra, cudaStream_t st) {
  const size_t smem = ((size_t)(len + 2 * halo + 8) * sizeof(float) + 15) & ~(size_t)15;
  if (ensure_smem((const void *)select_topk_resident_kernel<MODE>, smem))
    return cuda_failure(cudaErrorInvalidValue, "select kernel: shared memory");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(heads * CL));
  cfg.blockDim = dim3(NTC);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)CL;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, select_topk_resident_kernel<MODE>, z, T, k, recent,
                                           sink, len, idx, ra);
  if (e != cudaSuccess) return cuda_failure(e, "select kernel");
  return launch_status();
}

}  // namespace

int launch_select_topk(const float *z, int B, int H, int T, int k, int recent, int sink,
                       int32_t *idx, cudaStream_t st) {
  const long heads = (long)B * H;
  int CL, len;
  resident_plan(T - recent - sink, k - recent - sink, &CL, &len);
  if (len > 0 && heads * CL <= 0x7FFFFFFFL)
    return launch_resident<0>(z, heads, T, k, recent, sink, CL, len, 0, idx, RefineArgs{}, st);
  select_topk_kernel<<<(unsigned)heads, NT, 0, st>>>(z, T, k, recent, sink, idx);
  return launch_status();
}

bool hubkv_select_needs_z(int T, int k, int recent, int sink) {
  int CL, len;
  resident_plan(T - recent - sink, k - recent - sink, &CL, &len);
  return len == 0;
}

int launch_hubkv_select(const float *s, int B, int H, int T, int pool_width, float gamma, float r,
                        float beta_lo, float beta_hi, int flags, int k, int recent, int sink,
                        int32_t *idx, float *z_out, float *beta_out, void *ws,
                        const RefinePlan &plan, float *z_tmp, cudaStream_t st) {
  const long heads = (long)B * H;
  const int half = pool_width / 2;
  int rc = launch_refine_beta(s, B, H, T, beta_lo, beta_hi, flags, beta_out, ws, plan, st);
  if (rc != KV_OK) return rc;
  const float *beta_ws = reinterpret_cast<const float *>(static_cast<const char *>(ws) + plan.beta_offset);
  int CL, len;
  resident_plan(T - recent - sink, k - recent - sink, &CL, &len);
  if (len > 0 && heads * CL <= 0x7FFFFFFFL) {
    RefineArgs ra{beta_ws, z_out, gamma, r * r, half};
    if (flags & KV_HUB_AVGPOOL)
      return launch_resident<2>(s, heads, T, k, recent, sink, CL, len, half, idx, ra, st);
    return launch_resident<1>(s, heads, T, k, recent, sink, CL, len, half, idx, ra, st);
  }
  // too long to hold a head on chip (or everything kept): z first, then the
  // streaming selection
  float *z = z_out ? z_out : z_tmp;
  rc = launch_refine_apply(s, B, H, T, half, gamma, r, flags, beta_ws, z, st);
  if (rc != KV_OK) return rc;
  select_topk_kernel<<<(unsigned)heads, NT, 0, st>>>(z, T, k, recent, sink, idx);
  return launch_status();
}

}  // namespace kvc
