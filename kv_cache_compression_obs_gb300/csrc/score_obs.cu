// score_obs.cu -- observation-window attention mass per cached token (CUDA-core path).
//
// Computes, for every unit (b, KV head h) and prompt key j,
//     s[b][h][j] = sum over the G query heads of the group and the W window rows
//                  (prompt position p = T-W+w, keys j <= p) of softmax_j(scale q.k_j),
// the accumulated attention of the H2O page (观察二) taken over SnapKV's
// observation window (KV-cache blog §4.3) with the 1/sqrt(d_head) softmax of
// blog §1.1.  The column sum needs every row's softmax normaliser, which needs
// every key, so the work runs in three launches:
//   1. stats:   per (row block, key split) the running max m and sum Z of
//               2^(x - m), x = scale*log2(e)*q.k, over the split's keys;
//   2. combine: per row M = max m and 1/Z with Z = sum Z_s 2^(m_s - M);
//   3. colsum:  per key block, sum over rows of 2^(x - M) / Z.
// Logits are computed twice (once per pass) in fp32 FMA with 64x64 shared-memory
// tiles; the sums are fixed-order, so repeated runs give identical bits.  This is
// the path for fp32 inputs; bf16 inputs go to the tensor-core kernel of
// score_obs_tc.cu.
#include <cmath>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int RB = 64;   // query rows per tile
constexpr int KT = 64;   // keys per tile
constexpr int NT = 256;  // threads: 16 row groups x 16 key groups, 4x4 logits each
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTargetCtas = 4 * kNumSmsHint;

// Stage `rows` rows (row0..row0+rows-1) of a [*][D] slab into shared memory as
// float, row stride D+1 (the +1 keeps column reads conflict-free); rows at or
// beyond `valid` are zero-filled.
template <typename T, int D>
__device__ __forceinline__ void stage_rows(float *dst, const T *src, long row0, int valid, int rows) {
  constexpr int N = Vec16<T>::N;
  constexpr int VPR = D / N;
  for (int e = threadIdx.x; e < rows * VPR; e += NT) {
    const int r = e / VPR, v = e % VPR;
    float f[N];
    if (r < valid) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(src + (row0 + r) * D + v * N));
      Vec16<T>::unpack(raw, f);
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i) f[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < N; ++i) dst[r * (D + 1) + v * N + i] = f[i];
  }
}

// Largest prompt position among window rows r0 .. r0+n-1 (row r sits at T-W+(r%W)).
__device__ __forceinline__ int block_max_pos(int r0, int n, int T, int W) {
  if (n >= W || (r0 % W) + n - 1 >= W) return T - 1;
  return T - W + (r0 % W) + n - 1;
}

// acc[a][i] = <Qs row ty*4+a, Ks row tx+16i>
template <int D>
__device__ __forceinline__ void tile_dots(const float *Qs, const float *Ks, int ty, int tx,
                                          float acc[4][4]) {
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[a][i] = 0.f;
#pragma unroll 8
  for (int c = 0; c < D; ++c) {
    float q[4], k[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) q[a] = Qs[(ty * 4 + a) * (D + 1) + c];
#pragma unroll
    for (int i = 0; i < 4; ++i) k[i] = Ks[(tx + 16 * i) * (D + 1) + c];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[a][i] = fmaf(q[a], k[i], acc[a][i]);
  }
}

template <typename T, int D>
__global__ __launch_bounds__(NT) void score_stats_kernel(
    const T *__restrict__ Q, const T *__restrict__ K, int Hq, int Hkv, int Tlen, int W, int gw,
    int row_blocks, float scale_log2, int split_len, int n_splits, float2 *__restrict__ part) {
  extern __shared__ float sm[];
  float *Qs = sm;
  float *Ks = sm + RB * (D + 1);
  const long flat = blockIdx.x;
  const int rb = static_cast<int>(flat % row_blocks);
  const int split = static_cast<int>((flat / row_blocks) % n_splits);
  const long unit = flat / ((long)row_blocks * n_splits);
  const int G = Hq / Hkv;
  const long b = unit / Hkv;
  const int h = static_cast<int>(unit % Hkv);
  const int r0 = rb * RB;
  const int nrows = min(RB, gw - r0);
  const T *Qu = Q + ((b * Hq + (long)h * G) * W) * D;
  const T *Ku = K + unit * (long)Tlen * D;
  stage_rows<T, D>(Qs, Qu, r0, nrows, RB);

  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const unsigned gmask = 0xFFFFu << (16 * (ty & 1));  // the 16 lanes sharing ty
  int prow[4];
  float m[4], z[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int r = r0 + ty * 4 + a;
    prow[a] = (r < gw) ? Tlen - W + (r % W) : -1;
    m[a] = -INFINITY;
    z[a] = 0.f;
  }
  const int j_begin = split * split_len;
  const int j_stop = min(min(Tlen, j_begin + split_len), block_max_pos(r0, nrows, Tlen, W) + 1);
  for (int j0 = j_begin; j0 < j_stop; j0 += KT) {
    __syncthreads();
    stage_rows<T, D>(Ks, Ku, j0, min(KT, j_stop - j0), KT);
    __syncthreads();
    float acc[4][4];
    tile_dots<D>(Qs, Ks, ty, tx, acc);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      float x[4], tmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = j0 + tx + 16 * i;
        x[i] = (j < j_stop && j <= prow[a]) ? acc[a][i] * scale_log2 : -INFINITY;
        tmax = fmaxf(tmax, x[i]);
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(gmask, tmax, off));
      const float mnew = fmaxf(m[a], tmax);
      float zt = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) zt += (x[i] == -INFINITY) ? 0.f : exp2f(x[i] - mnew);
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) zt += __shfl_xor_sync(gmask, zt, off);
      const float rescale = (m[a] == -INFINITY) ? 0.f : exp2f(m[a] - mnew);
      z[a] = z[a] * rescale + zt;
      m[a] = mnew;
    }
  }
  if (tx == 0) {
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int r = r0 + ty * 4 + a;
      if (r < gw) part[(unit * n_splits + split) * gw + r] = make_float2(m[a], z[a]);
    }
  }
}

}  // namespace

__global__ void score_combine_kernel(const float2 *__restrict__ part, int n_splits, int gw,
                                     long total_rows, float2 *__restrict__ fin) {
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total_rows) return;
  const long unit = i / gw;
  const int r = static_cast<int>(i % gw);
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, part[(unit * n_splits + s) * gw + r].x);
  float Z = 0.f;
  for (int s = 0; s < n_splits; ++s) {
    const float2 p = part[(unit * n_splits + s) * gw + r];
    if (p.x != -INFINITY) Z += p.y * exp2f(p.x - M);
  }
  fin[i] = make_float2(M, 1.0f / Z);  // every row sees key 0, so Z >= 1
}

int launch_score_combine(const float2 *part, int n_splits, int gw, long rows, float2 *fin,
                         cudaStream_t st) {
  score_combine_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, st>>>(part, n_splits, gw, rows, fin);
  return launch_status();
}

namespace {

template <typename T, int D>
__global__ __launch_bounds__(NT) void score_colsum_kernel(
    const T *__restrict__ Q, const T *__restrict__ K, int Hq, int Hkv, int Tlen, int W, int gw,
    int key_blocks, float scale_log2, const float2 *__restrict__ fin, float *__restrict__ s_out) {
  extern __shared__ float sm[];
  float *Ks = sm;
  float *Qs = sm + KT * (D + 1);
  float2 *st = reinterpret_cast<float2 *>(Qs + RB * (D + 1));
  const long flat = blockIdx.x;
  const int kb = static_cast<int>(flat % key_blocks);
  const long unit = flat / key_blocks;
  const int G = Hq / Hkv;
  const long b = unit / Hkv;
  const int h = static_cast<int>(unit % Hkv);
  const T *Qu = Q + ((b * Hq + (long)h * G) * W) * D;
  const T *Ku = K + unit * (long)Tlen * D;
  const int j0 = kb * KT;
  const int nkeys = min(KT, Tlen - j0);
  stage_rows<T, D>(Ks, Ku, j0, nkeys, KT);

  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  float colacc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int r0 = 0; r0 < gw; r0 += RB) {
    const int nrows = min(RB, gw - r0);
    if (block_max_pos(r0, nrows, Tlen, W) < j0) continue;  // no row here sees these keys
    __syncthreads();
    stage_rows<T, D>(Qs, Qu, r0, nrows, RB);
    if (threadIdx.x < RB)
      st[threadIdx.x] = (threadIdx.x < nrows) ? fin[unit * gw + r0 + threadIdx.x]
                                              : make_float2(0.f, 0.f);
    __syncthreads();
    float acc[4][4];
    tile_dots<D>(Qs, Ks, ty, tx, acc);
    float blk[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int r = r0 + ty * 4 + a;
      if (r >= gw) continue;
      const int p = Tlen - W + (r % W);
      const float2 mz = st[ty * 4 + a];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = j0 + tx + 16 * i;
        if (j < Tlen && j <= p) blk[i] += exp2f(acc[a][i] * scale_log2 - mz.x) * mz.y;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) colacc[i] += blk[i];
  }
  __syncthreads();
  float *red = Qs;  // [16][KT]
#pragma unroll
  for (int i = 0; i < 4; ++i) red[ty * KT + tx + 16 * i] = colacc[i];
  __syncthreads();
  if (threadIdx.x < KT && threadIdx.x < nkeys) {
    float sum = 0.f;
    for (int g = 0; g < 16; ++g) sum += red[g * KT + threadIdx.x];
    s_out[unit * (long)Tlen + j0 + threadIdx.x] = sum;
  }
}

template <typename T, int D>
int run_score(const void *Q, const void *K, int B, int Hq, int Hkv, int Tlen, int W, float scale,
              float *s, void *ws, const ScorePlan &plan, cudaStream_t st) {
  const long units = (long)B * Hkv;
  float2 *part = static_cast<float2 *>(ws);
  float2 *fin = part + units * plan.n_splits * plan.gw;
  const float scale_log2 = scale * kLog2e;
  const size_t smem_stats = (size_t)(RB + KT) * (D + 1) * sizeof(float);
  const size_t smem_col = (size_t)(RB + KT) * (D + 1) * sizeof(float) + RB * sizeof(float2);
  if (ensure_smem((const void *)score_stats_kernel<T, D>, smem_stats) ||
      ensure_smem((const void *)score_colsum_kernel<T, D>, smem_col))
    return KV_ERR_CUDA;
  const long n1 = units * plan.row_blocks * plan.n_splits;
  score_stats_kernel<T, D><<<(unsigned)n1, NT, smem_stats, st>>>(
      static_cast<const T *>(Q), static_cast<const T *>(K), Hq, Hkv, Tlen, W, plan.gw,
      plan.row_blocks, scale_log2, plan.split_len, plan.n_splits, part);
  const long rows = units * plan.gw;
  score_combine_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, st>>>(part, plan.n_splits,
                                                                      plan.gw, rows, fin);
  const int key_blocks = (Tlen + KT - 1) / KT;
  score_colsum_kernel<T, D><<<(unsigned)(units * key_blocks), NT, smem_col, st>>>(
      static_cast<const T *>(Q), static_cast<const T *>(K), Hq, Hkv, Tlen, W, plan.gw, key_blocks,
      scale_log2, fin, s);
  return launch_status(3);
}

}  // namespace

// Split T into n pieces of a multiple of 128 keys, n about `want` (at least 1).
static void split_keys(int T, long want, int *n, int *len) {
  const int max_splits = (T + 127) / 128;
  if (want < 1) want = 1;
  if (want > max_splits) want = max_splits;
  const int per = (int)((T + want - 1) / want);
  *len = ((per + 127) / 128) * 128;
  *n = (T + *len - 1) / *len;
}

ScorePlan plan_score(int B, int Hq, int Hkv, int T, int W) {
  ScorePlan p{};
  p.gw = (Hq / Hkv) * W;
  p.row_blocks = (p.gw + RB - 1) / RB;
  const long units = (long)B * Hkv;
  const long base = units * p.row_blocks;
  split_keys(T, (kTargetCtas + base - 1) / (base > 0 ? base : 1), &p.n_splits, &p.split_len);
  const size_t core = (size_t)units * (p.n_splits + 1) * p.gw * sizeof(float2);
  const size_t tcb = tc_layout(B, Hq, Hkv, T, W).bytes;
  p.ws_bytes = core > tcb ? core : tcb;
  return p;
}

int launch_score_obs(const void *Q, const void *K, int B, int Hq, int Hkv, int T, int d, int W,
                     float scale, int dtype, float *s, void *ws, const ScorePlan &plan,
                     int *status, cudaStream_t st) {
  if (score_tc_eligible(dtype, d, Hq, Hkv, W))
    return launch_score_obs_tc(Q, K, B, Hq, Hkv, T, d, W, scale, s, ws, plan, status, st);
  if (dtype == KV_BF16) {
    if (d == 128) return run_score<__nv_bfloat16, 128>(Q, K, B, Hq, Hkv, T, W, scale, s, ws, plan, st);
    return run_score<__nv_bfloat16, 64>(Q, K, B, Hq, Hkv, T, W, scale, s, ws, plan, st);
  }
  if (d == 128) return run_score<float, 128>(Q, K, B, Hq, Hkv, T, W, scale, s, ws, plan, st);
  return run_score<float, 64>(Q, K, B, Hq, Hkv, T, W, scale, s, ws, plan, st);
}

}  // namespace kvc
