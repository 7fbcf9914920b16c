// h2o_decode.cu -- one H2O decode step over a preallocated slot cache.
//
// H2O page: 问题形式化 (|S_i| = k, at most one eviction per step, attention
// renormalised over the kept keys), 贪心驱逐算法 (Algorithm 1: accumulate the
// softmax into a per-token score, evict the lowest), 双缓冲 (the recent window
// is protected), FlexGen 改造 (the evicted slot is overwritten in place; the
// score vector is updated as a by-product of the attention kernel).
//
// Two launches per step:
//   stream -- one CTA per (unit, chunk of CH rows), where a unit is (b, KV head)
//             and its rows are the filled slots plus the new token.  The CTA
//             reads its K rows (one row per thread, the whole row's 16-byte loads
//             in flight, q from shared memory) into logits l_gj = scale <q_g, k_j>,
//             which it also writes to the workspace; takes its local max m_c and
//             normaliser Z_c per query head; and reads its V rows (one row per
//             warp, the lanes across d, 128 bytes per lane in flight) into its
//             output share o_c relative to m_c.  No CTA waits for another, so the
//             K and V streams of many CTAs overlap freely on every SM.
//   evict  -- one cluster of CE CTAs per unit: combines the chunks' (m_c, Z_c,
//             o_c) into the step's output; turns the stored logits into
//             probabilities, adds them to the slots' accumulators and takes each
//             CTA's (acc, pos)-smallest slot outside the recent window; after a
//             cluster barrier CTA 0 picks the smallest over the cluster (and the
//             new token itself when recent == 0) and appends the new token or
//             writes it over the victim; a last barrier keeps the CTAs' shared
//             memory alive until CTA 0 has read it.
// Workspace: the logits [units][G][cap+1], the chunks' (m, Z) [units][NCH][G] and
// output shares [units][NCH][G][D], all float.
#include <cmath>
#include <type_traits>

#include <cooperative_groups.h>

#include "kvc_internal.cuh"

namespace cg = cooperative_groups;

namespace kvc {
namespace {

constexpr int NT = 256;   // stream kernel threads
constexpr int NWARP = NT / 32;
constexpr int CH = 512;   // rows per stream CTA
constexpr int NTE = 256;  // evict kernel threads per CTA
constexpr int CE = 4;     // evict kernel CTAs per unit (one thread-block cluster)
constexpr int NWE = NTE / 32;

__device__ __forceinline__ bool better(float a, int p, float ba, int bp) {
  return a < ba || (a == ba && p < bp);
}

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

struct Ws {      // workspace carve-up
  float *lgw;    // [units][G][cap+1] logits
  float2 *mz;    // [units][nch][G] chunk max and normaliser
  float *opart;  // [units][nch][G][D] chunk output shares
};

__host__ __device__ inline int n_chunks(int cap) { return (cap + 1 + CH - 1) / CH; }

inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

Ws carve(void *ws, long units, int G, int cap) {
  Ws w;
  char *p = static_cast<char *>(ws);
  const size_t lg_bytes = align256((size_t)units * G * (cap + 1) * 4);
  const size_t mz_bytes = align256((size_t)units * n_chunks(cap) * G * 8);
  w.lgw = reinterpret_cast<float *>(p);
  w.mz = reinterpret_cast<float2 *>(p + lg_bytes);
  w.opart = reinterpret_cast<float *>(p + lg_bytes + mz_bytes);
  return w;
}

template <typename T, int D, int G>
__global__ __launch_bounds__(NT, 4) void decode_stream_kernel(
    const T *__restrict__ q, const T *__restrict__ k_new, const T *__restrict__ v_new,
    const T *__restrict__ Kc, const T *__restrict__ Vc, const int32_t *__restrict__ len, int Hq,
    int Hkv, int cap, float scale, int alg1, Ws ws, int *__restrict__ dev_status) {
  constexpr int EPL = Vec16<T>::N;              // elements per 16-byte vector
  constexpr int VPR = D * (int)sizeof(T) / 16;  // 16-byte vectors per K row
  constexpr int VB = VPR < 8 ? VPR : 8;         // K vectors per load batch
  constexpr int EV = D / 32;                    // V elements per lane
  using RV = RawV<T, EV>;
  constexpr int U = 128 / RV::BYTES;            // V rows per warp in flight (128 bytes per lane)
  __shared__ __align__(16) float qs[G * D];
  __shared__ float wst[NWARP * G];
  __shared__ float cst[G];
  extern __shared__ __align__(16) float dyn[];  // stream_smem_bytes(G, D)
  float *wred = dyn;                            // [NWARP][G][D]
  float *lg = dyn + NWARP * G * D;              // [CH][G] logits, then weights exp(l - m_c)

  const int nch = n_chunks(cap);
  const long unit = blockIdx.x / nch;
  const int c = static_cast<int>(blockIdx.x % nch);
  const long b = unit / Hkv;
  const int h = static_cast<int>(unit % Hkv);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = len[unit];
  if (n < 0 || n > cap) {
    if (c == 0 && threadIdx.x == 0 && dev_status) atomicExch(dev_status, (int)KV_ERR_INVALID_ARG);
    return;
  }
  const int nc = n + (alg1 ? 0 : 1);          // attended rows: slots 0..n-1, then the new token
  const int r0 = c * CH;
  const int nl = max(0, min(CH, nc - r0));    // this CTA's rows
  float2 *mz = ws.mz + (unit * nch + c) * G;
  float *op = ws.opart + (unit * nch + c) * (long)G * D;
  if (nl == 0) {
    if (threadIdx.x < G) mz[threadIdx.x] = make_float2(-INFINITY, 0.f);
    return;
  }

  const T *qg = q + (b * Hq + (long)h * G) * D;
  for (int t = threadIdx.x; t < G * D; t += NT) qs[t] = to_f32(qg[t]);
  __syncthreads();

  const T *Ku = Kc + unit * (long)cap * D;
  const T *Vu = Vc + unit * (long)cap * D;
  const T *kn = k_new + unit * (long)D;
  const T *vn = v_new + unit * (long)D;
  auto row_ptr = [&](const T *base, const T *fresh, int r) -> const T * {
    const int j = r0 + r;
    return (j < n) ? base + (long)j * D : fresh;
  };
  float *lgu = ws.lgw + unit * (long)G * (cap + 1);

  // 1. logits: one thread per row; two packed partial sums per query head
  for (int r = threadIdx.x; r < nl; r += NT) {
    const uint4 *row = reinterpret_cast<const uint4 *>(row_ptr(Ku, kn, r));
    float2 part[G];
#pragma unroll
    for (int g = 0; g < G; ++g) part[g] = make_float2(0.f, 0.f);
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
            part[g] = __ffma2_rn(make_float2(f[4 * e4 + 0], f[4 * e4 + 1]), make_float2(qq.x, qq.y), part[g]);
            part[g] = __ffma2_rn(make_float2(f[4 * e4 + 2], f[4 * e4 + 3]), make_float2(qq.z, qq.w), part[g]);
          }
        }
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float l = scale * (part[g].x + part[g].y);
      lg[r * G + g] = l;
      lgu[(long)g * (cap + 1) + r0 + r] = l;
    }
  }
  __syncthreads();

  // 2. the chunk's max, weights exp(l - m_c) and normaliser
  float mx[G];
#pragma unroll
  for (int g = 0; g < G; ++g) mx[g] = -INFINITY;
  for (int r = threadIdx.x; r < nl; r += NT)
#pragma unroll
    for (int g = 0; g < G; ++g) mx[g] = fmaxf(mx[g], lg[r * G + g]);
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xFFFFFFFFu, mx[g], off));
    if (lane == 0) wst[warp * G + g] = mx[g];
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float m = -INFINITY;
    for (int w = 0; w < NWARP; ++w) m = fmaxf(m, wst[w * G + threadIdx.x]);
    cst[threadIdx.x] = m;
  }
  __syncthreads();
  float zs[G];
#pragma unroll
  for (int g = 0; g < G; ++g) zs[g] = 0.f;
  for (int r = threadIdx.x; r < nl; r += NT)
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float e = expf(lg[r * G + g] - cst[g]);
      lg[r * G + g] = e;
      zs[g] += e;
    }
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) zs[g] += __shfl_xor_sync(0xFFFFFFFFu, zs[g], off);
  }
  __syncthreads();  // every thread is done reading wst (the max) before it is reused
  if (lane == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) wst[warp * G + g] = zs[g];
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float z = 0.f;
    for (int w = 0; w < NWARP; ++w) z += wst[w * G + threadIdx.x];
    mz[threadIdx.x] = make_float2(cst[threadIdx.x], z);
  }

  // 3. the chunk's output share relative to m_c: one V row per warp, lanes across d
  static_assert(EV % 2 == 0, "V elements per lane come in pairs");
  float2 o[G][EV / 2];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < EV / 2; ++e) o[g][e] = make_float2(0.f, 0.f);
  for (int rr = warp * U; rr < nl; rr += NWARP * U) {
    typename RV::Word raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (rr + u < nl) raw[u] = RV::load(row_ptr(Vu, vn, rr + u) + lane * EV);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (rr + u < nl) {
        float vv[EV];
        RV::unpack(raw[u], vv);
        float pg[G];
#pragma unroll
        for (int g = 0; g < G; ++g) pg[g] = lg[(rr + u) * G + g];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < EV / 2; ++e)
            o[g][e] = __ffma2_rn(make_float2(pg[g], pg[g]), make_float2(vv[2 * e], vv[2 * e + 1]), o[g][e]);
      }
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < EV / 2; ++e) {
      wred[(warp * G + g) * D + lane * EV + 2 * e] = o[g][e].x;
      wred[(warp * G + g) * D + lane * EV + 2 * e + 1] = o[g][e].y;
    }
  __syncthreads();
  for (int t = threadIdx.x; t < G * D; t += NT) {
    float s = 0.f;
    for (int w = 0; w < NWARP; ++w) s += wred[w * G * D + t];
    op[t] = s;
  }
}

struct Cand {
  float acc;
  int pos;
  int slot;       // -2: no candidate
  float accself;  // the new token's score, from the CTA that holds its row
};

template <int G, int D>
__global__ __launch_bounds__(NTE) void decode_evict_kernel(
    int32_t *__restrict__ pos, float *__restrict__ acc, int32_t *__restrict__ len, int Hq,
    int Hkv, int cap, int recent, int new_pos, int alg1, Ws ws, void *__restrict__ Kc,
    void *__restrict__ Vc, const void *__restrict__ k_new, const void *__restrict__ v_new,
    int row_bytes, float *__restrict__ o_out, int32_t *__restrict__ evicted,
    int *__restrict__ dev_status) {
  constexpr int RU = 4;  // rows per thread in flight
  __shared__ float gm[G], gz[G];
  __shared__ Cand wc[NWE];
  __shared__ Cand cand;
  __shared__ int sh_slot;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const long unit = blockIdx.x / CE;
  const long b = unit / Hkv;
  const int h = static_cast<int>(unit % Hkv);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = len[unit];
  if (n < 0 || n > cap) return;  // same n in the whole cluster; reported by the stream kernel
  const int nch = n_chunks(cap);
  const int nc = n + (alg1 ? 0 : 1);
  const float2 *mz = ws.mz + unit * nch * G;
  const int nuse = (nc + CH - 1) / CH;  // chunks that hold rows
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    float m = -INFINITY;
    for (int c = 0; c < nuse; ++c) m = fmaxf(m, mz[c * G + g].x);
    float z = 0.f;
    for (int c = 0; c < nuse; ++c) {
      const float2 p = mz[c * G + g];
      if (p.x != -INFINITY) z += p.y * expf(p.x - m);
    }
    gm[g] = m;
    gz[g] = z;
  }
  __syncthreads();
  // this CTA's part of the output: o_g = sum_c o_c exp(m_c - m) / Z
  float *ou = o_out + (b * Hq + (long)h * G) * D;
  const float *opu = ws.opart + unit * nch * (long)G * D;
  constexpr int GD = G * D;
  for (int t = rank * (GD / CE) + threadIdx.x; t < (rank + 1) * (GD / CE); t += NTE) {
    const int g = t / D;
    float s = 0.f;
    for (int c = 0; c < nuse; ++c) {
      const float mc = mz[c * G + g].x;
      if (mc != -INFINITY) s += opu[(long)c * GD + t] * expf(mc - gm[g]);
    }
    ou[t] = nuse ? s / gz[g] : 0.f;
  }
  // this CTA's rows: probabilities -> accumulators, eviction candidate
  const int per = (nc + CE - 1) / CE;
  const int j0 = min(nc, rank * per), j1 = min(nc, j0 + per);
  const float *lgu = ws.lgw + unit * (long)G * (cap + 1);
  float *au = acc + unit * (long)cap;
  int32_t *pu = pos + unit * (long)cap;
  const long lim = (long)new_pos - recent;
  float best_a = INFINITY;
  int best_p = 0x7FFFFFFF, best_j = -2;
  float acc_self = 0.f;
  for (int jb = j0 + threadIdx.x; jb < j1; jb += RU * NTE) {
    float lv[RU][G], av[RU];
    int pv[RU];
#pragma unroll
    for (int u = 0; u < RU; ++u) {
      const int j = jb + u * NTE;
      if (j < j1) {
#pragma unroll
        for (int g = 0; g < G; ++g) lv[u][g] = lgu[(long)g * (cap + 1) + j];
        if (j < n) {
          av[u] = au[j];
          pv[u] = pu[j];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < RU; ++u) {
      const int j = jb + u * NTE;
      if (j >= j1) continue;
      float P = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g) P += expf(lv[u][g] - gm[g]) / gz[g];
      if (j < n) {
        const float a = av[u] + P;
        au[j] = a;
        if ((long)pv[u] <= lim && better(a, pv[u], best_a, best_p)) {
          best_a = a;
          best_p = pv[u];
          best_j = j;
        }
      } else {
        acc_self = P;  // the new token
      }
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
  if (lane == 0) wc[warp] = Cand{best_a, best_p, best_j, acc_self};
  __syncthreads();
  if (threadIdx.x == 0) {
    Cand c{INFINITY, 0x7FFFFFFF, -2, 0.f};
    for (int w = 0; w < NWE; ++w) {
      if (wc[w].slot != -2 && (c.slot == -2 || better(wc[w].acc, wc[w].pos, c.acc, c.pos))) {
        c.acc = wc[w].acc;
        c.pos = wc[w].pos;
        c.slot = wc[w].slot;
      }
      c.accself += wc[w].accself;
    }
    cand = c;
  }
  cluster.sync();  // #1: every CTA's candidate is visible
  if (rank == 0) {
    if (threadIdx.x == 0) {
      float ba = INFINITY, accnew = 0.f;
      int bp = 0x7FFFFFFF, bj = -2;
      for (int r = 0; r < CE; ++r) {
        const Cand cc = *cluster.map_shared_rank(&cand, r);
        if (cc.slot != -2 && (bj == -2 || better(cc.acc, cc.pos, ba, bp))) {
          ba = cc.acc;
          bp = cc.pos;
          bj = cc.slot;
        }
        accnew += cc.accself;
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
      evicted[unit] = ev;
      if (slot >= 0) {
        pu[slot] = new_pos;
        au[slot] = accnew;
      }
    }
    __syncthreads();
    const int slot = sh_slot;
    if (slot >= 0) {
      const int vecs = row_bytes / 16;
      uint4 *kd = reinterpret_cast<uint4 *>(static_cast<char *>(Kc) + (unit * (long)cap + slot) * row_bytes);
      uint4 *vd = reinterpret_cast<uint4 *>(static_cast<char *>(Vc) + (unit * (long)cap + slot) * row_bytes);
      const uint4 *ks = reinterpret_cast<const uint4 *>(static_cast<const char *>(k_new) + unit * (long)row_bytes);
      const uint4 *vs = reinterpret_cast<const uint4 *>(static_cast<const char *>(v_new) + unit * (long)row_bytes);
      for (int t = threadIdx.x; t < vecs; t += NTE) {
        kd[t] = __ldg(ks + t);
        vd[t] = __ldg(vs + t);
      }
    }
  }
  cluster.sync();  // #2: rank 0 has finished reading the others' shared memory
}

constexpr size_t stream_smem_bytes(int G, int D) { return (size_t)(NWARP * G * D + G * CH) * sizeof(float); }

template <typename T, int D, int G>
int run_decode(const void *q, const void *k_new, const void *v_new, void *K_cache, void *V_cache,
               int32_t *pos, float *acc, int32_t *len, int B, int Hq, int Hkv, int cap,
               int recent, int new_pos, float scale, int flags, void *workspace, float *o,
               int32_t *evicted, int *dev_status, cudaStream_t st) {
  const long units = (long)B * Hkv;
  const Ws ws = carve(workspace, units, G, cap);
  const int alg1 = (flags & KV_H2O_ALG1) ? 1 : 0;
  const size_t smem = stream_smem_bytes(G, D);
  if (ensure_smem((const void *)decode_stream_kernel<T, D, G>, smem)) return KV_ERR_CUDA;
  decode_stream_kernel<T, D, G><<<(unsigned)(units * n_chunks(cap)), NT, smem, st>>>(
      static_cast<const T *>(q), static_cast<const T *>(k_new), static_cast<const T *>(v_new),
      static_cast<const T *>(K_cache), static_cast<const T *>(V_cache), len, Hq, Hkv, cap, scale,
      alg1, ws, dev_status);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units * CE), 1, 1);
  cfg.blockDim = dim3(NTE, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CE;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_evict_kernel<G, D>, pos, acc, len, Hq, Hkv, cap, recent,
                         new_pos, alg1, ws, K_cache, V_cache, k_new, v_new, D * (int)sizeof(T), o,
                         evicted, dev_status) != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  return launch_status(2);
}

template <typename T, int D>
int dispatch_g(int G, const void *q, const void *k_new, const void *v_new, void *K_cache,
               void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq, int Hkv,
               int cap, int recent, int new_pos, float scale, int flags, void *workspace,
               float *o, int32_t *evicted, int *dev_status, cudaStream_t st) {
#define KVC_DEC(GG)                                                                          \
  if (G == GG)                                                                               \
    return run_decode<T, D, GG>(q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq, Hkv, \
                                cap, recent, new_pos, scale, flags, workspace, o, evicted,    \
                                dev_status, st);
  KVC_DEC(1)
  KVC_DEC(2)
  KVC_DEC(4)
  KVC_DEC(8)
#undef KVC_DEC
  return KV_ERR_UNSUPPORTED;
}

}  // namespace

size_t decode_workspace_bytes(long units, int G, int cap, int d) {
  const size_t lg_bytes = align256((size_t)units * G * (cap + 1) * 4);
  const size_t mz_bytes = align256((size_t)units * n_chunks(cap) * G * 8);
  const size_t op_bytes = (size_t)units * n_chunks(cap) * G * d * 4;
  return lg_bytes + mz_bytes + op_bytes;
}

int launch_decode_step(const void *q, const void *k_new, const void *v_new, void *K_cache,
                       void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq,
                       int Hkv, int cap, int d, int recent, int32_t new_pos, float scale,
                       int flags, int dtype, void *workspace, float *o, int32_t *evicted,
                       int *dev_status, cudaStream_t st) {
  const int G = Hq / Hkv;
  if (dtype == KV_BF16) {
    if (d == 128)
      return dispatch_g<__nv_bfloat16, 128>(G, q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq,
                                            Hkv, cap, recent, new_pos, scale, flags, workspace, o,
                                            evicted, dev_status, st);
    return dispatch_g<__nv_bfloat16, 64>(G, q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq,
                                         Hkv, cap, recent, new_pos, scale, flags, workspace, o,
                                         evicted, dev_status, st);
  }
  if (d == 128)
    return dispatch_g<float, 128>(G, q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq, Hkv,
                                  cap, recent, new_pos, scale, flags, workspace, o, evicted,
                                  dev_status, st);
  return dispatch_g<float, 64>(G, q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq, Hkv,
                               cap, recent, new_pos, scale, flags, workspace, o, evicted,
                               dev_status, st);
}

}  // namespace kvc
