// hubkv_refine.cu -- HubKV score refinement (HubKV walkthrough, Method: 最终算法).
//
//   1. local hubs: M_i = max_{|j-i| <= pool_width/2} s_j, hub iff s_i == M_i;
//   2. SMD discount: q_i = s_i for hubs, gamma s_i otherwise;
//   3. head weight: sel_h = 1 - H_h / ln T with H_h the entropy of s_h / sum(s_h);
//      beta_h = clip(sel_h / mean over the batch row's heads, lo, hi), 1 if mean 0;
//   4. ratio gate: z_i = s_i + r^2 (beta_h q_i - s_i).
// Three launches: an entropy reduction per (head, chunk) writing fixed-order
// partial sums; one block per batch row turning them into beta_h (double
// precision, fixed order, so the result is reproducible bit for bit); one pass
// that applies steps 1, 2 and 4 with a shared-memory halo for the pooling window.
#include <cmath>

#include "kvc_internal.cuh"
#include "refine_common.cuh"

namespace kvc {
namespace {

constexpr int NT = 256;
constexpr int kChunk = 16384;      // entropy chunk (elements): 64 per thread
constexpr int kApply = 2048;       // elements per block of the apply pass
constexpr int kMaxHalo = 64;       // pool_width <= 129

// Neumaier-compensated float sum.
struct CSum {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float t = s + x;
    c += (fabsf(s) >= fabsf(x)) ? (s - t) + x : (x - t) + s;
    s = t;
  }
  __device__ __forceinline__ double value() const { return (double)s + (double)c; }
};

// Per (head, chunk): sum s and sum s ln s (0 ln 0 = 0), reduced in a fixed order
// (per thread, then a warp butterfly in double, then the warps in order).  ln s
// comes from the SFU's base-2 logarithm times ln 2 (relative error about 1e-7
// for the scores' range, far below what the head weights need).  A chunk's
// scores move as 16-byte vectors, four a thread in flight, when the head's row
// is 16-byte aligned; otherwise as scalars.
__global__ __launch_bounds__(NT) void refine_entropy_kernel(const float *__restrict__ s, int T,
                                                            int n_chunks,
                                                            double2 *__restrict__ part) {
  const long head = blockIdx.x / n_chunks;
  const int chunk = blockIdx.x % n_chunks;
  const float *sv = s + head * (long)T;
  const int i0 = chunk * kChunk, i1 = min(T, i0 + kChunk);
  CSum a, c;
  auto add = [&](float x) {
    a.add(x);
    if (x > 0.f) c.add(x * (__log2f(x) * 0.69314718f));
  };
  if ((reinterpret_cast<uintptr_t>(sv + i0) & 15) == 0) {
    const int n4 = (i1 - i0) >> 2;
    const float4 *v4 = reinterpret_cast<const float4 *>(sv + i0);
    for (int base = threadIdx.x; base < n4; base += 4 * NT) {
      float4 x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = base + u * NT;
        x[u] = j < n4 ? __ldg(v4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        add(x[u].x);
        add(x[u].y);
        add(x[u].z);
        add(x[u].w);
      }
    }
    for (int i = i0 + 4 * n4 + threadIdx.x; i < i1; i += NT) add(__ldg(sv + i));
  } else {
    for (int base = i0 + threadIdx.x; base < i1; base += 4 * NT) {
      float x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {  // four loads in flight per thread
        const int i = base + u * NT;
        x[u] = i < i1 ? __ldg(sv + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) add(x[u]);
    }
  }
  double ra = a.value(), rc = c.value();
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ra += __shfl_xor_sync(0xFFFFFFFFu, ra, o);
    rc += __shfl_xor_sync(0xFFFFFFFFu, rc, o);
  }
  __shared__ double wa[NT / 32], wc[NT / 32];
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    wa[warp] = ra;
    wc[warp] = rc;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double sa = 0.0, sc = 0.0;
    for (int w = 0; w < NT / 32; ++w) {
      sa += wa[w];
      sc += wc[w];
    }
    part[head * n_chunks + chunk] = make_double2(sa, sc);
  }
}

// One block per batch row: sel_h per head in double (fixed chunk order), the row
// mean in head order, then beta_h.
__global__ void refine_beta_kernel(const double2 *__restrict__ part, int H, int T, int n_chunks,
                                   float beta_lo, float beta_hi, int fixed_head,
                                   float *__restrict__ beta_ws, float *__restrict__ beta_out) {
  extern __shared__ double sel[];
  const long b = blockIdx.x;
  const double lnT = log((double)T);
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    double S = 0.0, C = 0.0;
    for (int c = 0; c < n_chunks; ++c) {
      const double2 p = part[(b * H + h) * n_chunks + c];
      S += p.x;
      C += p.y;
    }
    sel[h] = (T > 1 && S > 0.0) ? 1.0 - (log(S) - C / S) / lnT : 0.0;
  }
  __syncthreads();
  __shared__ double mean;
  if (threadIdx.x == 0) {
    double acc = 0.0;
    for (int h = 0; h < H; ++h) acc += sel[h];
    mean = acc / H;
  }
  __syncthreads();
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    double bt = 1.0;  // also the fixed head weight of the KV_HUB_FIXED_HEAD variant
    if (mean != 0.0 && !fixed_head) bt = fmin(fmax(sel[h] / mean, (double)beta_lo), (double)beta_hi);
    beta_ws[b * H + h] = (float)bt;
    if (beta_out) beta_out[b * H + h] = (float)bt;
  }
}

template <bool AVG>
__global__ __launch_bounds__(NT) void refine_apply_kernel(
    const float *__restrict__ s, int T, int blocks_per_head, int half, float gamma, float r2,
    const float *__restrict__ beta_ws, float *__restrict__ z) {
  extern __shared__ __align__(16) float tile_raw[];
  const long head = blockIdx.x / blocks_per_head;
  const int blk = blockIdx.x % blocks_per_head;
  const float beta = beta_ws[head];
  const float *sv = s + head * (long)T;
  float *zv = z + head * (long)T;
  const int i0 = blk * kApply, i1 = min(T, i0 + kApply);
  const int lo = i0 - half, n = (i1 - i0) + 2 * half;
  // tile[t] = s[lo + t] (-inf past the prompt's ends), placed `toff` floats into
  // the buffer so that it has the global addresses' 16-byte phase: the aligned
  // middle moves as 16-byte vectors, the ragged ends as scalars
  const int rmis = (int)((reinterpret_cast<uintptr_t>(sv) >> 2) & 3);
  const int toff = (((rmis + lo) % 4) + 4) % 4;
  float *tile = tile_raw + toff;
  {
    const int c0 = max(lo, 0), c1 = min(lo + n, T);
    const int a0 = min(c1, c0 + (4 - (rmis + c0) % 4) % 4);
    const int e0 = max(a0, c1 - (rmis + c1) % 4);
    const int n4 = (e0 - a0) >> 2;
    const float4 *g4 = reinterpret_cast<const float4 *>(sv + a0);
    float4 *t4 = reinterpret_cast<float4 *>(tile + (a0 - lo));
    for (int j = threadIdx.x; j < n4; j += NT) t4[j] = __ldg(g4 + j);
    const int front = a0 - lo, back = lo + n - e0;
    for (int t = threadIdx.x; t < front + back; t += NT) {
      const int tt = t < front ? t : (e0 - lo) + (t - front);
      const int i = lo + tt;
      tile[tt] = (i >= 0 && i < T) ? __ldg(sv + i) : -INFINITY;
    }
  }
  __syncthreads();
  if (!AVG && half == 2) {
    // local hubs over a window of 5, four consecutive candidates a thread: the 8
    // scores around them give the four window maxima from shared pair maxima
    // (the same values as hub_gate: a maximum does not depend on its order)
    const bool vec = ((reinterpret_cast<uintptr_t>(zv + i0)) & 15) == 0;
    for (int c = i0 + 4 * threadIdx.x; c < i1; c += 4 * NT) {
      const float *w = tile + (c - 2 - lo);  // s of positions c-2 .. c+5
      float x[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) x[q] = w[q];
      const float m01 = fmaxf(x[0], x[1]), m23 = fmaxf(x[2], x[3]), m45 = fmaxf(x[4], x[5]),
                  m67 = fmaxf(x[6], x[7]);
      const float M[4] = {fmaxf(fmaxf(m01, m23), x[4]), fmaxf(fmaxf(x[1], m23), m45),
                          fmaxf(fmaxf(m23, m45), x[6]), fmaxf(fmaxf(x[3], m45), m67)};
      float zq[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float si = x[q + 2];
        const float qi = (si == M[q]) ? si : gamma * si;
        zq[q] = fmaf(r2, fmaf(beta, qi, -si), si);
      }
      if (vec && c + 4 <= i1) {
        *reinterpret_cast<float4 *>(zv + c) = make_float4(zq[0], zq[1], zq[2], zq[3]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (c + q < i1) zv[c + q] = zq[q];
      }
    }
  } else {
    for (int i = i0 + threadIdx.x; i < i1; i += NT)
      zv[i] = hub_gate<AVG>(tile + (i - lo), half, i, T, gamma, r2, beta);
  }
}

}  // namespace

RefinePlan plan_refine(int B, int H, int T) {
  RefinePlan p{};
  p.chunk = kChunk;
  p.n_chunks = (T + kChunk - 1) / kChunk;
  p.beta_offset = ((size_t)B * H * p.n_chunks * sizeof(double2) + 255) / 256 * 256;
  p.ws_bytes = p.beta_offset + (size_t)B * H * sizeof(float);
  return p;
}

int launch_refine_beta(const float *s, int B, int H, int T, float beta_lo, float beta_hi, int flags,
                       float *beta, void *ws, const RefinePlan &plan, cudaStream_t st) {
  const long heads = (long)B * H;
  double2 *part = static_cast<double2 *>(ws);
  float *beta_ws = reinterpret_cast<float *>(static_cast<char *>(ws) + plan.beta_offset);
  refine_entropy_kernel<<<(unsigned)(heads * plan.n_chunks), NT, 0, st>>>(s, T, plan.n_chunks, part);
  const int bt = H < 256 ? ((H + 31) / 32) * 32 : 256;
  refine_beta_kernel<<<(unsigned)B, bt, (size_t)H * sizeof(double), st>>>(
      part, H, T, plan.n_chunks, beta_lo, beta_hi, (flags & KV_HUB_FIXED_HEAD) ? 1 : 0, beta_ws, beta);
  return launch_status(2);
}

int launch_refine_apply(const float *s, int B, int H, int T, int half, float gamma, float r, int flags,
                        const float *beta_ws, float *z, cudaStream_t st) {
  const long heads = (long)B * H;
  const int bph = (T + kApply - 1) / kApply;
  const size_t smem = (size_t)(kApply + 2 * half + 16) * sizeof(float);
  if (flags & KV_HUB_AVGPOOL)
    refine_apply_kernel<true><<<(unsigned)(heads * bph), NT, smem, st>>>(s, T, bph, half, gamma, r * r,
                                                                      beta_ws, z);
  else
    refine_apply_kernel<false><<<(unsigned)(heads * bph), NT, smem, st>>>(s, T, bph, half, gamma, r * r,
                                                                       beta_ws, z);
  return launch_status(1);
}

int launch_hubkv_refine(const float *s, int B, int H, int T, int pool_width, float gamma,
                        float r, float beta_lo, float beta_hi, int flags, float *z, float *beta,
                        void *ws, const RefinePlan &plan, cudaStream_t st) {
  const int half = pool_width / 2;
  if (half > kMaxHalo) return KV_ERR_UNSUPPORTED;
  const int rc = launch_refine_beta(s, B, H, T, beta_lo, beta_hi, flags, beta, ws, plan, st);
  if (rc != KV_OK) return rc;
  const float *beta_ws = reinterpret_cast<const float *>(static_cast<const char *>(ws) + plan.beta_offset);
  return launch_refine_apply(s, B, H, T, half, gamma, r, flags, beta_ws, z, st);
}

}  // namespace kvc
