// h2o_decode.cu -- one H2O decode step over a preallocated slot cache.
//
// H2O page: 问题形式化 (|S_i| = k, at most one eviction per step, attention
// renormalised over the kept keys), 贪心驱逐算法 (Algorithm 1: accumulate the
// softmax into a per-token score, evict the lowest), 双缓冲 (the recent window
// is protected), FlexGen 改造 (the evicted slot is overwritten in place, the
// score vector is updated as a by-product of the attention kernel).
//
// One block per unit (b, KV head) serves the G query heads of the group:
//   1. logits l_gj = scale <q_g, k_j> over the filled slots (+ the new token),
//      a group of lanes per 16-byte-vectorised K row (coalesced), kept in smem;
//   2. per g the max and the normaliser (fixed-order block reductions);
//   3. p_gj = exp(l_gj - m_g) / Z_g; acc_j += sum_g p_gj; the block-wide argmin of
//      (acc, pos) over the eviction candidates;
//   4. o_g = sum_j p_gj v_j with V read once, reduced across warps in a fixed order;
//   5. the new token is appended, or written over the victim's slot.
// The block never waits on another block.
#include <cmath>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int NT = 256;
constexpr int NWARP = NT / 32;

__device__ __forceinline__ bool better(float a, int p, float ba, int bp) {
  return a < ba || (a == ba && p < bp);
}

template <typename T, int D, int G>
__global__ __launch_bounds__(NT) void decode_kernel(
    const T *__restrict__ q, const T *__restrict__ k_new, const T *__restrict__ v_new,
    T *__restrict__ Kc, T *__restrict__ Vc, int32_t *__restrict__ pos, float *__restrict__ acc,
    int32_t *__restrict__ len, int Hq, int Hkv, int cap, int recent, int new_pos, float scale,
    int alg1, float *__restrict__ o_out, int32_t *__restrict__ evicted,
    int *__restrict__ dev_status) {
  constexpr int EPL = Vec16<T>::N;             // elements per 16-byte vector
  constexpr int LPR = D / EPL;                 // lanes per row
  constexpr int RPW = 32 / LPR;                // rows per warp per iteration
  constexpr int NG = NWARP * RPW;              // row groups per block
  extern __shared__ float sm[];
  float *qs = sm;                               // [G][D]
  float *red = qs + G * D;                      // [NWARP][G][D]
  float *stat = red + NWARP * G * D;            // [2][G] (max, 1/Z) + scratch
  float *lg = stat + 4 * G + 2 * NWARP * G + 4 * NWARP;  // [G][cap+1] logits -> probabilities
  float *wred = stat + 4 * G;                   // [NWARP][G] per-warp partials
  int *wpos = reinterpret_cast<int *>(wred + NWARP * G);   // [NWARP] argmin pos
  float *wacc = reinterpret_cast<float *>(wpos + NWARP);   // [NWARP] argmin acc
  int *widx = reinterpret_cast<int *>(wacc + NWARP);       // [NWARP] argmin slot
  int *wmisc = reinterpret_cast<int *>(widx + NWARP);      // [NWARP]

  const long unit = blockIdx.x;
  const long b = unit / Hkv;
  const int h = static_cast<int>(unit % Hkv);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = len[unit];
  if (n < 0 || n > cap) {
    if (threadIdx.x == 0 && dev_status) atomicExch(dev_status, (int)KV_ERR_INVALID_ARG);
    return;
  }
  const int with_self = alg1 ? 0 : 1;
  const int nc = n + with_self;
  const int ldl = cap + 1;
  const T *qg = q + (b * Hq + (long)h * G) * D;
  for (int t = threadIdx.x; t < G * D; t += NT) qs[t] = to_f32(qg[t]);
  __syncthreads();

  const T *Ku = Kc + unit * (long)cap * D;
  const T *Vu = Vc + unit * (long)cap * D;
  const T *kn = k_new + unit * (long)D;
  const T *vn = v_new + unit * (long)D;
  const int sl = lane % LPR;   // lane within the row group
  const int rg = lane / LPR;   // row group within the warp

  // 1. logits
  for (int j0 = warp * RPW; j0 < nc; j0 += NG) {
    const int j = j0 + rg;
    float f[EPL];
    if (j < nc) {
      const T *row = (j < n) ? Ku + (long)j * D : kn;
      Vec16<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(row) + sl), f);
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) f[e] = 0.f;
    }
    float part[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) a = fmaf(f[e], qs[g * D + sl * EPL + e], a);
      part[g] = a;
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1)
#pragma unroll
      for (int g = 0; g < G; ++g) part[g] += __shfl_xor_sync(0xFFFFFFFFu, part[g], off);
    if (sl == 0 && j < nc) {
#pragma unroll
      for (int g = 0; g < G; ++g) lg[g * ldl + j] = scale * part[g];
    }
  }
  __syncthreads();

  // 2. max and normaliser per query head
  float mx[G];
#pragma unroll
  for (int g = 0; g < G; ++g) mx[g] = -INFINITY;
  for (int j = threadIdx.x; j < nc; j += NT)
#pragma unroll
    for (int g = 0; g < G; ++g) mx[g] = fmaxf(mx[g], lg[g * ldl + j]);
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xFFFFFFFFu, mx[g], off));
    if (lane == 0) wred[warp * G + g] = mx[g];
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float m = -INFINITY;
    for (int w = 0; w < NWARP; ++w) m = fmaxf(m, wred[w * G + threadIdx.x]);
    stat[threadIdx.x] = m;
  }
  __syncthreads();
  float zs[G];
#pragma unroll
  for (int g = 0; g < G; ++g) zs[g] = 0.f;
  for (int j = threadIdx.x; j < nc; j += NT)
#pragma unroll
    for (int g = 0; g < G; ++g) zs[g] += expf(lg[g * ldl + j] - stat[g]);
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) zs[g] += __shfl_xor_sync(0xFFFFFFFFu, zs[g], off);
    if (lane == 0) wred[warp * G + g] = zs[g];
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float z = 0.f;
    for (int w = 0; w < NWARP; ++w) z += wred[w * G + threadIdx.x];
    stat[G + threadIdx.x] = z;
  }
  __syncthreads();

  // 3. probabilities, accumulator update, eviction candidate
  const long lim = (long)new_pos - recent;
  float best_a = INFINITY;
  int best_p = 0x7FFFFFFF, best_j = -2;
  float acc_self = 0.f;
  float *au = acc + unit * (long)cap;
  int32_t *pu = pos + unit * (long)cap;
  for (int j = threadIdx.x; j < nc; j += NT) {
    float P = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float p = expf(lg[g * ldl + j] - stat[g]) / stat[G + g];
      lg[g * ldl + j] = p;
      P += p;
    }
    if (j < n) {
      const float a = au[j] + P;
      au[j] = a;
      const int pj = pu[j];
      if ((long)pj <= lim && better(a, pj, best_a, best_p)) {
        best_a = a;
        best_p = pj;
        best_j = j;
      }
    } else {
      acc_self = P;  // j == n: the new token (only when it attends itself)
    }
  }
  // the new token's accumulator (0 under Algorithm 1) is needed by every thread
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
    wacc[warp] = best_a;
    wpos[warp] = best_p;
    widx[warp] = best_j;
    wmisc[warp] = __float_as_int(acc_self);
  }
  __syncthreads();

  // 4. attention output o_g = sum_j p_gj v_j
  float op_[G][EPL];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < EPL; ++e) op_[g][e] = 0.f;
  for (int j0 = warp * RPW; j0 < nc; j0 += NG) {
    const int j = j0 + rg;
    if (j < nc) {
      float f[EPL];
      const T *row = (j < n) ? Vu + (long)j * D : vn;
      Vec16<T>::unpack(__ldg(reinterpret_cast<const uint4 *>(row) + sl), f);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float p = lg[g * ldl + j];
#pragma unroll
        for (int e = 0; e < EPL; ++e) op_[g][e] = fmaf(p, f[e], op_[g][e]);
      }
    }
  }
#pragma unroll
  for (int off = LPR; off < 32; off <<= 1)
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < EPL; ++e) op_[g][e] += __shfl_xor_sync(0xFFFFFFFFu, op_[g][e], off);
  if (rg == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < EPL; ++e) red[(warp * G + g) * D + sl * EPL + e] = op_[g][e];
  }
  __syncthreads();
  float *ou = o_out + (b * Hq + (long)h * G) * D;
  for (int t = threadIdx.x; t < G * D; t += NT) {
    float s = 0.f;
    for (int w = 0; w < NWARP; ++w) s += red[w * G * D + t];
    ou[t] = s;
  }

  // 5. append or overwrite (all reads of K, V, acc and pos are done)
  __shared__ int sh_slot, sh_evicted;
  __shared__ float sh_accnew;
  if (threadIdx.x == 0) {
    float accnew = 0.f;
    for (int w = 0; w < NWARP; ++w) accnew += __int_as_float(wmisc[w]);  // one warp holds it
    float ba = INFINITY;
    int bp = 0x7FFFFFFF, bj = -2;
    for (int w = 0; w < NWARP; ++w) {
      if (widx[w] != -2 && (bj == -2 || better(wacc[w], wpos[w], ba, bp))) {
        ba = wacc[w];
        bp = wpos[w];
        bj = widx[w];
      }
    }
    int slot = -1, ev = -1;
    if (n < cap) {
      slot = n;
      len[unit] = n + 1;
    } else {
      if (recent == 0 && (bj == -2 || better(accnew, new_pos, ba, bp))) bj = -1;  // the new token
      if (bj == -2) {
        if (dev_status) atomicExch(dev_status, (int)KV_ERR_INVALID_ARG);
      } else if (bj == -1) {
        ev = new_pos;
      } else {
        slot = bj;
        ev = bp;
      }
    }
    sh_slot = slot;
    sh_accnew = accnew;
    sh_evicted = ev;
    evicted[unit] = ev;
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
    if (threadIdx.x == 0) {
      pu[slot] = new_pos;
      au[slot] = sh_accnew;
    }
  }
}

template <typename T, int D, int G>
int run_decode(const void *q, const void *k_new, const void *v_new, void *K_cache, void *V_cache,
               int32_t *pos, float *acc, int32_t *len, int B, int Hq, int Hkv, int cap,
               int recent, int new_pos, float scale, int flags, float *o, int32_t *evicted,
               int *dev_status, cudaStream_t st) {
  const size_t smem = decode_smem_bytes(G, cap, D);
  if (ensure_smem((const void *)decode_kernel<T, D, G>, smem)) return KV_ERR_UNSUPPORTED;
  const long units = (long)B * Hkv;
  decode_kernel<T, D, G><<<(unsigned)units, NT, smem, st>>>(
      static_cast<const T *>(q), static_cast<const T *>(k_new), static_cast<const T *>(v_new),
      static_cast<T *>(K_cache), static_cast<T *>(V_cache), pos, acc, len, Hq, Hkv, cap, recent,
      new_pos, scale, (flags & KV_H2O_ALG1) ? 1 : 0, o, evicted, dev_status);
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
  const size_t floats = (size_t)G * d + (size_t)NWARP * G * d + 4 * G + 2 * NWARP * G + 4 * NWARP +
                        (size_t)G * (cap + 1);
  return floats * sizeof(float);
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
