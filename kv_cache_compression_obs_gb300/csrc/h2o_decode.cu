// h2o_decode.cu -- one H2O decode step over a preallocated slot cache.
//
// H2O page: 问题形式化 (|S_i| = k, at most one eviction per step, attention
// renormalised over the kept keys), 贪心驱逐算法 (Algorithm 1: accumulate the
// softmax into a per-token score, evict the lowest), 双缓冲 (the recent window
// is protected), FlexGen 改造 (the evicted slot is overwritten in place; the
// score vector is updated as a by-product of the attention kernel).
//
// One thread-block cluster of C CTAs per unit (b, KV head); CTA r owns slot
// range r of the unit (CTA 0 also owns the new token) and serves the G query
// heads of the group:
//   1. logits l_gj = scale <q_g, k_j> over its rows, one thread per K row with the
//      whole row's 16-byte loads in flight, kept in shared memory;
//   2. its local max and normaliser per g; cluster barrier; every CTA combines
//      the C local pairs, read through distributed shared memory in rank order,
//      into the same global (m_g, Z_g);
//   3. p_gj = exp(l_gj - m_g) / Z_g; acc_j += sum_g p_gj; its (acc, pos)-smallest
//      eviction candidate; its share of o_g = sum_j p_gj v_j (V read once, one
//      row per warp with the lanes across d, sixteen rows per warp in flight);
//   4. cluster barrier; CTA 0 takes the smallest candidate over the cluster (and
//      the new token itself when recent == 0), sums the o shares in rank order,
//      and appends the new token or writes it over the victim's slot;
//   5. a last cluster barrier keeps every CTA's shared memory alive until CTA 0
//      has read it.
// The cluster barriers are hardware barriers that every CTA reaches
// unconditionally; no CTA spins on memory written by another.
#include <cooperative_groups.h>

#include <cmath>
#include <type_traits>

#include "kvc_internal.cuh"

namespace cg = cooperative_groups;

namespace kvc {
namespace {

constexpr int NT = 256;
constexpr int NWARP = NT / 32;
constexpr int kMaxCluster = 5;
constexpr int kSlotsPerCta = 1300;  // target rows per CTA when choosing the cluster size

__device__ __forceinline__ bool better(float a, int p, float ba, int bp) {
  return a < ba || (a == ba && p < bp);
}

struct Cand {
  float acc;
  int pos;
  int slot;  // -2 = no candidate
  int pad;
};

template <int G, int D>
struct Layout {
  // floats, in order: qs[G*D], opart[G*D], wred[NWARP*G*D], stat[2G], wstat[NWARP*G], lg[G*ldl]
  static constexpr int QS = 0;
  static constexpr int OPART = QS + G * D;
  static constexpr int WRED = OPART + G * D;
  static constexpr int STAT = WRED + NWARP * G * D;
  static constexpr int WSTAT = STAT + 2 * G;
  static constexpr int CAND = WSTAT + NWARP * G;           // Cand (4 words)
  static constexpr int WCAND = CAND + 4;                   // NWARP x Cand
  static constexpr int MISC = WCAND + 4 * NWARP;           // acc_new, slot, evicted, ...
  static constexpr int LG = MISC + 8;
  // after lg: the rows' accumulators and positions, staged at kernel start
  static size_t bytes(int ldl) { return (size_t)(LG + G * ldl + 2 * ldl) * sizeof(float); }
};

// EV consecutive elements of a row held packed (EV * sizeof(T) = 4, 8 or 16 bytes)
// until they are used, so that many rows can be in flight per thread.
template <typename T, int EV>
struct RawV {
  static constexpr int BYTES = EV * (int)sizeof(T);
  using Word = typename std::conditional<BYTES == 16, uint4,
               typename std::conditional<BYTES == 8, uint2, uint32_t>::type>::type;
  __device__ __forceinline__ static Word load(const T *p) { return __ldg(reinterpret_cast<const Word *>(p)); }
  __device__ __forceinline__ static void unpack(const Word &w, float (&f)[EV]) {
    if constexpr (BYTES == 16) {
      Vec16<T>::unpack(w, f);
    } else if constexpr (BYTES == 8 && sizeof(T) == 2) {
      f[0] = __uint_as_float(w.x << 16);
      f[1] = __uint_as_float(w.x & 0xFFFF0000u);
      f[2] = __uint_as_float(w.y << 16);
      f[3] = __uint_as_float(w.y & 0xFFFF0000u);
    } else if constexpr (BYTES == 8) {
      f[0] = __uint_as_float(w.x);
      f[1] = __uint_as_float(w.y);
    } else {
      f[0] = __uint_as_float(w << 16);
      f[1] = __uint_as_float(w & 0xFFFF0000u);
    }
  }
};

template <typename T, int D, int G>
__global__ __launch_bounds__(NT) void decode_kernel(
    const T *__restrict__ q, const T *__restrict__ k_new, const T *__restrict__ v_new,
    T *__restrict__ Kc, T *__restrict__ Vc, int32_t *__restrict__ pos, float *__restrict__ acc,
    int32_t *__restrict__ len, int Hq, int Hkv, int cap, int recent, int new_pos, float scale,
    int alg1, int C, int ldl, float *__restrict__ o_out, int32_t *__restrict__ evicted,
    int *__restrict__ dev_status) {
  using L = Layout<G, D>;
  constexpr int EPL = Vec16<T>::N;  // elements per 16-byte vector
  constexpr int LPR = D / EPL;      // lanes per row
  constexpr int RPW = 32 / LPR;     // rows per warp per iteration
  constexpr int NG = NWARP * RPW;   // row groups per block
  extern __shared__ float sm[];
  float *qs = sm + L::QS;
  float *opart = sm + L::OPART;
  float *wred = sm + L::WRED;
  float *stat = sm + L::STAT;
  float *wstat = sm + L::WSTAT;
  Cand *cand = reinterpret_cast<Cand *>(sm + L::CAND);
  Cand *wcand = reinterpret_cast<Cand *>(sm + L::WCAND);
  float *misc = sm + L::MISC;
  float *lg = sm + L::LG;

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const long unit = blockIdx.x / C;
  const long b = unit / Hkv;
  const int h = static_cast<int>(unit % Hkv);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = len[unit];
  if (n < 0 || n > cap) {  // same n in every CTA of the cluster: all leave before any barrier
    if (rank == 0 && threadIdx.x == 0 && dev_status) atomicExch(dev_status, (int)KV_ERR_INVALID_ARG);
    return;
  }
  const int with_self = alg1 ? 0 : 1;
  const int chunk = (n + C - 1) / C;
  const int j0 = min(n, rank * chunk);
  const int j1 = min(n, j0 + chunk);
  const int self_here = (with_self && rank == 0) ? 1 : 0;
  const int nl = (j1 - j0) + self_here;  // local rows; row nl-1 is the new token when self_here
  float *sacc = lg + G * ldl;                             // [ldl] accumulators of rows j0..j1-1
  int *spos = reinterpret_cast<int *>(sacc + ldl);        // [ldl] their positions
  float *au = acc + unit * (long)cap;
  int32_t *pu = pos + unit * (long)cap;
  // The accumulators and positions are needed only after the K pass: copy them
  // to shared memory asynchronously now so that their latency hides behind it.
  for (int r = threadIdx.x; r < j1 - j0; r += NT) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(sacc + r)),
                 "l"(au + j0 + r)
                 : "memory");
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(spos + r)),
                 "l"(pu + j0 + r)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");

  const T *qg = q + (b * Hq + (long)h * G) * D;
  for (int t = threadIdx.x; t < G * D; t += NT) qs[t] = to_f32(qg[t]);
  __syncthreads();

  const T *Ku = Kc + unit * (long)cap * D;
  const T *Vu = Vc + unit * (long)cap * D;
  const T *kn = k_new + unit * (long)D;
  const T *vn = v_new + unit * (long)D;
  const int sl = lane % LPR;  // lane within the row group
  const int rg = lane / LPR;  // row group within the warp
  auto row_ptr = [&](const T *base, const T *fresh, int r) -> const T * {
    return (r < j1 - j0) ? base + (long)(j0 + r) * D : fresh;
  };

  // 1. logits: one thread per row, the whole row requested before use (VPR
  //    16-byte loads in flight per thread), q read from shared memory (broadcast)
  constexpr int VPR = D * (int)sizeof(T) / 16;   // 16-byte vectors per row
  constexpr int VB = VPR < 8 ? VPR : 8;          // vectors per batch
  for (int r = threadIdx.x; r < nl; r += NT) {
    const uint4 *row = reinterpret_cast<const uint4 *>(row_ptr(Ku, kn, r));
    float part[G];
#pragma unroll
    for (int g = 0; g < G; ++g) part[g] = 0.f;
#pragma unroll
    for (int v0 = 0; v0 < VPR; v0 += VB) {
      uint4 raw[VB];
#pragma unroll
      for (int v = 0; v < VB; ++v) raw[v] = __ldg(row + v0 + v);
#pragma unroll
      for (int v = 0; v < VB; ++v) {
        float f[EPL];
        Vec16<T>::unpack(raw[v], f);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 *q4 = reinterpret_cast<const float4 *>(qs + g * D + (v0 + v) * EPL);
#pragma unroll
          for (int e4 = 0; e4 < EPL / 4; ++e4) {
            const float4 qq = q4[e4];
            part[g] = fmaf(f[4 * e4 + 0], qq.x, part[g]);
            part[g] = fmaf(f[4 * e4 + 1], qq.y, part[g]);
            part[g] = fmaf(f[4 * e4 + 2], qq.z, part[g]);
            part[g] = fmaf(f[4 * e4 + 3], qq.w, part[g]);
          }
        }
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) lg[g * ldl + r] = scale * part[g];
  }
  __syncthreads();

  // 2. local max and normaliser per query head, then the cluster-wide pair
  float mx[G];
#pragma unroll
  for (int g = 0; g < G; ++g) mx[g] = -INFINITY;
  for (int r = threadIdx.x; r < nl; r += NT)
#pragma unroll
    for (int g = 0; g < G; ++g) mx[g] = fmaxf(mx[g], lg[g * ldl + r]);
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xFFFFFFFFu, mx[g], off));
    if (lane == 0) wstat[warp * G + g] = mx[g];
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float m = -INFINITY;
    for (int w = 0; w < NWARP; ++w) m = fmaxf(m, wstat[w * G + threadIdx.x]);
    stat[threadIdx.x] = m;
  }
  __syncthreads();
  float zs[G];
#pragma unroll
  for (int g = 0; g < G; ++g) zs[g] = 0.f;
  for (int r = threadIdx.x; r < nl; r += NT)
#pragma unroll
    for (int g = 0; g < G; ++g) zs[g] += expf(lg[g * ldl + r] - stat[g]);
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) zs[g] += __shfl_xor_sync(0xFFFFFFFFu, zs[g], off);
    if (lane == 0) wstat[warp * G + g] = zs[g];
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float z = 0.f;
    for (int w = 0; w < NWARP; ++w) z += wstat[w * G + threadIdx.x];
    stat[G + threadIdx.x] = z;  // stat = [m_0..m_G-1, Z_0..Z_G-1] of this CTA
  }
  cluster.sync();  // #1: every CTA's local pair is visible
  __shared__ float gm[8], gz[8];
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    float m = -INFINITY;
    for (int c = 0; c < C; ++c) m = fmaxf(m, cluster.map_shared_rank(stat, c)[g]);
    float z = 0.f;
    for (int c = 0; c < C; ++c) {
      const float *st = cluster.map_shared_rank(stat, c);
      if (st[g] != -INFINITY) z += st[G + g] * expf(st[g] - m);
    }
    gm[g] = m;
    gz[g] = z;
  }
  __syncthreads();

  // 3. probabilities, accumulators, this CTA's eviction candidate
  const long lim = (long)new_pos - recent;
  float best_a = INFINITY;
  int best_p = 0x7FFFFFFF, best_j = -2;
  float acc_self = 0.f;
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  for (int r = threadIdx.x; r < nl; r += NT) {
    float P = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float p = expf(lg[g * ldl + r] - gm[g]) / gz[g];
      lg[g * ldl + r] = p;
      P += p;
    }
    if (r < j1 - j0) {
      const int j = j0 + r;
      const float a = sacc[r] + P;
      au[j] = a;
      const int pj = spos[r];
      if ((long)pj <= lim && better(a, pj, best_a, best_p)) {
        best_a = a;
        best_p = pj;
        best_j = j;
      }
    } else {
      acc_self = P;  // the new token (CTA 0 only)
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc_self += __shfl_xor_sync(0xFFFFFFFFu, acc_self, off);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float oa = __shfl_xor_sync(0xFFFFFFFFu, best_a, off);
    const int op = __shfl_xor_sync(0xFFFFFFFFu, best_p, off);
    const int oj = __shfl_xor_sync(0xFFFFFFFFu, best_j, off);
    if (oj != -2 && (best_j == -2 || better(oa, op, best_a, best_p))) {
      best_a = oa;
      best_p = op;
      best_j = oj;
    }
  }
  if (lane == 0) {
    wcand[warp] = Cand{best_a, best_p, best_j, 0};
    wstat[warp * G] = acc_self;  // (reuse) per-warp share of the new token's score
  }
  __syncthreads();

  // o share: sum over this CTA's rows of p_gj v_j.  One row per warp at a time,
  // the lanes across d (EV elements each), 16 rows per warp in flight.
  constexpr int EV = D / 32;
  using RV = RawV<T, EV>;
  constexpr int U = 128 / RV::BYTES;  // 128 bytes of V in flight per lane
  float op_[G][EV];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < EV; ++e) op_[g][e] = 0.f;
  for (int r0 = warp * U; r0 < nl; r0 += NWARP * U) {
    typename RV::Word raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (r0 + u < nl) raw[u] = RV::load(row_ptr(Vu, vn, r0 + u) + lane * EV);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (r0 + u < nl) {
        float vv[EV];
        RV::unpack(raw[u], vv);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float p = lg[g * ldl + r0 + u];
#pragma unroll
          for (int e = 0; e < EV; ++e) op_[g][e] = fmaf(p, vv[e], op_[g][e]);
        }
      }
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < EV; ++e) wred[(warp * G + g) * D + lane * EV + e] = op_[g][e];
  __syncthreads();
  for (int t = threadIdx.x; t < G * D; t += NT) {
    float s = 0.f;
    for (int w = 0; w < NWARP; ++w) s += wred[w * G * D + t];
    opart[t] = s;
  }
  if (threadIdx.x == 0) {
    Cand best{INFINITY, 0x7FFFFFFF, -2, 0};
    float accnew = 0.f;
    for (int w = 0; w < NWARP; ++w) {
      const Cand c = wcand[w];
      if (c.slot != -2 && (best.slot == -2 || better(c.acc, c.pos, best.acc, best.pos))) best = c;
      accnew += wstat[w * G];
    }
    *cand = best;
    misc[0] = accnew;
  }
  cluster.sync();  // #2: candidates and o shares of every CTA are visible

  // 4. CTA 0: the step's decision and output
  __shared__ int sh_slot;
  if (rank == 0) {
    float *ou = o_out + (b * Hq + (long)h * G) * D;
    for (int t = threadIdx.x; t < G * D; t += NT) {
      float s = 0.f;
      for (int c = 0; c < C; ++c) s += cluster.map_shared_rank(opart, c)[t];
      ou[t] = s;
    }
    if (threadIdx.x == 0) {
      Cand best{INFINITY, 0x7FFFFFFF, -2, 0};
      for (int c = 0; c < C; ++c) {
        const Cand cc = *cluster.map_shared_rank(cand, c);
        if (cc.slot != -2 && (best.slot == -2 || better(cc.acc, cc.pos, best.acc, best.pos))) best = cc;
      }
      const float accnew = misc[0];
      int slot = -1, ev = -1;
      if (n < cap) {
        slot = n;
        len[unit] = n + 1;
      } else {
        if (recent == 0 && (best.slot == -2 || better(accnew, new_pos, best.acc, best.pos)))
          best.slot = -1;  // the new token itself
        if (best.slot == -2) {
          if (dev_status) atomicExch(dev_status, (int)KV_ERR_INVALID_ARG);
        } else if (best.slot == -1) {
          ev = new_pos;
        } else {
          slot = best.slot;
          ev = best.pos;
        }
      }
      sh_slot = slot;
      evicted[unit] = ev;
      if (slot >= 0) {
        pu[slot] = new_pos;
        au[slot] = accnew;
      }
    }
    __syncthreads();
    const int slot = sh_slot;
    if (slot >= 0) {
      uint4 *kd = reinterpret_cast<uint4 *>(Kc + (unit * (long)cap + slot) * D);
      uint4 *vd = reinterpret_cast<uint4 *>(Vc + (unit * (long)cap + slot) * D);
      for (int t = threadIdx.x; t < LPR; t += NT) {
        kd[t] = __ldg(reinterpret_cast<const uint4 *>(kn) + t);
        vd[t] = __ldg(reinterpret_cast<const uint4 *>(vn) + t);
      }
    }
  }
  cluster.sync();  // #3: CTA 0 has finished reading the others' shared memory
}

int cluster_size_for(int cap) {
  int c = (cap + kSlotsPerCta - 1) / kSlotsPerCta;
  if (c < 1) c = 1;
  if (c > kMaxCluster) c = kMaxCluster;
  return c;
}

int ldl_for(int cap, int C) { return (cap + C - 1) / C + 1; }

template <typename T, int D, int G>
int run_decode(const void *q, const void *k_new, const void *v_new, void *K_cache, void *V_cache,
               int32_t *pos, float *acc, int32_t *len, int B, int Hq, int Hkv, int cap,
               int recent, int new_pos, float scale, int flags, float *o, int32_t *evicted,
               int *dev_status, cudaStream_t st) {
  const int C = cluster_size_for(cap);
  const int ldl = ldl_for(cap, C);
  const size_t smem = Layout<G, D>::bytes(ldl);
  if (ensure_smem((const void *)decode_kernel<T, D, G>, smem)) return KV_ERR_UNSUPPORTED;
  const long units = (long)B * Hkv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units * C), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, decode_kernel<T, D, G>, static_cast<const T *>(q), static_cast<const T *>(k_new),
      static_cast<const T *>(v_new), static_cast<T *>(K_cache), static_cast<T *>(V_cache), pos, acc,
      len, Hq, Hkv, cap, recent, new_pos, scale, (flags & KV_H2O_ALG1) ? 1 : 0, C, ldl, o, evicted,
      dev_status);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  return launch_status();
}

template <typename T, int D>
int dispatch_g(int G, const void *q, const void *k_new, const void *v_new, void *K_cache,
               void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq, int Hkv,
               int cap, int recent, int new_pos, float scale, int flags, float *o,
               int32_t *evicted, int *dev_status, cudaStream_t st) {
#define KVC_DEC(GG)                                                                          \
  if (G == GG)                                                                               \
    return run_decode<T, D, GG>(q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq, Hkv, \
                                cap, recent, new_pos, scale, flags, o, evicted, dev_status, st);
  KVC_DEC(1)
  KVC_DEC(2)
  KVC_DEC(4)
  KVC_DEC(8)
#undef KVC_DEC
  return KV_ERR_UNSUPPORTED;
}

}  // namespace

size_t decode_smem_bytes(int G, int cap, int d) {
  const int C = cluster_size_for(cap);
  const int ldl = ldl_for(cap, C);
  const size_t fixed = (size_t)G * d * (2 + NWARP) + 2 * G + NWARP * G + 4 + 4 * NWARP + 8;
  return (fixed + (size_t)G * ldl + 2 * (size_t)ldl) * sizeof(float);
}

int launch_decode_step(const void *q, const void *k_new, const void *v_new, void *K_cache,
                       void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq,
                       int Hkv, int cap, int d, int recent, int32_t new_pos, float scale,
                       int flags, int dtype, float *o, int32_t *evicted, int *dev_status,
                       cudaStream_t st) {
  const int G = Hq / Hkv;
  if (dtype == KV_BF16) {
    if (d == 128)
      return dispatch_g<__nv_bfloat16, 128>(G, q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq,
                                            Hkv, cap, recent, new_pos, scale, flags, o, evicted,
                                            dev_status, st);
    return dispatch_g<__nv_bfloat16, 64>(G, q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq,
                                         Hkv, cap, recent, new_pos, scale, flags, o, evicted,
                                         dev_status, st);
  }
  if (d == 128)
    return dispatch_g<float, 128>(G, q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq, Hkv,
                                  cap, recent, new_pos, scale, flags, o, evicted, dev_status, st);
  return dispatch_g<float, 64>(G, q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq, Hkv,
                               cap, recent, new_pos, scale, flags, o, evicted, dev_status, st);
}

}  // namespace kvc
