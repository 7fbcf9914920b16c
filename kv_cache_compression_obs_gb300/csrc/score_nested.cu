// score_nested.cu -- NestedKV key-only scoring (NestedKV technical summary,
// 1. Continuum Geheugentoestand and 2. Buitenste Leraar).
//
// Per unit (b, h) over its T keys, with kh_i = k_i / |k_i|:
//   a_s(i) = -cos(k_i, sum_j kh_j)                       stable anchor
//   a_e(i) = -cos(k_i, sum of kh over i's block)          episodic anchor, blocks of
//                                                         ceil(T / n_blocks) keys
//   a_c(i) = -cos(k_i, sum of kh over [i-window+1, i])    current anchor (causal)
//   D_k    = mean of the n_disc largest a_k - mean of the n_disc smallest
//   w      = softmax_k(D_k + log_prior_k)
//   score  = max_k a_k(i) if the std of the three a_k(i) exceeds thresh, else
//            sum_k w_k a_k(i).
// (A mean and a sum point the same way, so the anchors are kept as sums.)
//
// HBM-bound key scans on the CUDA cores, four launches:
//   1. anchors_kernel: one CTA of two warps per (unit, episodic block); each
//      warp runs two token streams over contiguous ranges (16 lanes per key,
//      features spread over the lanes; every stream first re-reads the window
//      before its range, so fewer, longer streams re-read less).  Each key is normalised once; the block sum of kh goes
//      to the workspace; the causal window sum is kept as P (the current
//      window-aligned chunk's prefix) + Q (the previous chunk's suffix, its
//      total minus the rows that left the window), so every running sum
//      restarts each `window` keys and rounding cannot drift; the rows leaving
//      the window are re-read and their 1/|k| comes from a per-stream ring in
//      shared memory.  A row's first read marks it evict_last in L2 and its
//      re-read evict_first: only the rows inside some stream's window (tens of
//      MB) are protected, so the re-reads hit L2 instead of HBM.  Packed f32x2
//      arithmetic throughout.  Writes a_c.
//   2. global_kernel: same grid; adds the unit's block sums into the stable
//      anchor, re-reads the block's keys (four lanes per key, the anchors'
//      slices in registers) and writes a_s and a_e.
//   3. disc_kernel: one CTA per (unit, scale): radix selects (order-preserving
//      32-bit keys) of the n_disc-th largest and smallest a_k sharing every pass,
//      then the two sums.
//   4. final_kernel: elementwise weights, surprise, routing.
// The window scan's per-token cross-lane sums go through batched butterflies
// over a stream's 16 lanes: V values of a batch's tokens reduce in
// V-1 + (4 - log2 V) shuffles instead of 4 V.
#include <type_traits>

#include "kvc_internal.cuh"
#include "select_common.cuh"
#include "tc_common.cuh"

namespace kvc {
namespace {

constexpr int NWARP = 4;  // warps per CTA of the global scan
constexpr int NT_SCAN = NWARP * 32;
constexpr int NT_DISC = 1024;

// ---- row loads: lane holds features P2*2*lane .. as P2 float2 pairs -----------
// Loads carry an L2 cache-policy operand (createpolicy): rows that will be read
// again soon are kept (evict_last), rows read for the last time go first.
template <int NW32> struct Words;
template <> struct Words<2> {
  __device__ __forceinline__ static void load(const void *p, uint64_t pol, uint32_t (&w)[2]) {
    asm("ld.global.nc.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
                 : "=r"(w[0]), "=r"(w[1]) : "l"(p), "l"(pol));
  }
};
template <> struct Words<4> {
  __device__ __forceinline__ static void load(const void *p, uint64_t pol, uint32_t (&w)[4]) {
    asm("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "l"(p), "l"(pol));
  }
};

template <typename T, int D> struct Row {
  static constexpr int F = D / 32;                          // features per lane
  static constexpr int P2 = F / 2;                          // float2 pairs per lane
  static constexpr int NW = F * (int)sizeof(T) / 4;         // 32-bit words per lane
  __device__ __forceinline__ static void load(const T *row, int lane, uint64_t pol, float2 (&x)[P2]) {
    uint32_t w[NW];
    Words<NW>::load(reinterpret_cast<const char *>(row) + lane * NW * 4, pol, w);
    if constexpr (sizeof(T) == 2) {  // bf16: a word holds two features
#pragma unroll
      for (int p = 0; p < P2; ++p)
        x[p] = make_float2(__uint_as_float(w[p] << 16), __uint_as_float(w[p] & 0xFFFF0000u));
    } else {
#pragma unroll
      for (int p = 0; p < P2; ++p) x[p] = make_float2(__uint_as_float(w[2 * p]), __uint_as_float(w[2 * p + 1]));
    }
  }
};

__device__ __forceinline__ float hsum(float2 a) { return a.x + a.y; }

// ---- 1. block sums and the current (moving-window) anchor ---------------------
// Sixteen lanes per key: a warp runs two independent token streams, lane l of a
// stream's group holding the features of pieces l, l+16, ... of each row (a
// group's load covers contiguous bytes of one row), so a token's sums take four
// shuffle levels instead of five and every shuffle serves two tokens.
constexpr int GW = 16;                // lanes per stream
constexpr int NSW = 32 / GW;          // streams per warp
constexpr int AWARP = 2;              // warps per CTA of the window scan
constexpr int NT_ANCH = AWARP * 32;
constexpr int NSTREAM = AWARP * NSW;  // streams per CTA
constexpr int NB = 4;                 // tokens of a stream per batch
constexpr int OWN = GW / NB;          // group lanes holding one token's sums after an NB-value reduction

template <typename T, int D> struct GroupRow {
  static constexpr int RB = D * (int)sizeof(T);       // bytes per row
  static constexpr int LB = RB / GW;                  // bytes per lane
  static constexpr int US = LB < 16 ? LB : 16;        // bytes per load
  static constexpr int NL = LB / US;                  // loads per lane
  static constexpr int PPL = US / (2 * (int)sizeof(T));  // float2 pairs per load
  static constexpr int P2 = NL * PPL;                 // float2 pairs per lane
  static_assert(RB % GW == 0 && LB % US == 0 && PPL >= 1, "row must split into pieces over the group");
  // feature of the first element of pair p held by group lane g
  __device__ __forceinline__ static int feature(int g, int p) {
    return ((US * GW) * (p / PPL) + US * g) / (int)sizeof(T) + 2 * (p % PPL);
  }
  __device__ __forceinline__ static void load(const T *row, int g, uint64_t pol, float2 (&x)[P2]) {
    const char *base = reinterpret_cast<const char *>(row) + US * g;
#pragma unroll
    for (int j = 0; j < NL; ++j) {
      uint32_t w[US / 4];
      Words<US / 4>::load(base + (US * GW) * j, pol, w);
      if constexpr (sizeof(T) == 2) {  // bf16: a word holds two features
#pragma unroll
        for (int e = 0; e < PPL; ++e)
          x[j * PPL + e] = make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
      } else {
#pragma unroll
        for (int e = 0; e < PPL; ++e)
          x[j * PPL + e] = make_float2(__uint_as_float(w[2 * e]), __uint_as_float(w[2 * e + 1]));
      }
    }
  }
};

// reduce_scatter over the GW lanes of a group: afterwards group lane g holds the
// total of value g / (GW / V) (V = 2, 4 or 8).
template <int V>
__device__ __forceinline__ float reduce_scatter_group(float (&v)[V], int g) {
  int count = V;
#pragma unroll
  for (int o = GW / 2; o >= 1; o >>= 1) {
    if (count > 1) {
      const int half = count >> 1;
      const bool up = (g & o) != 0;
#pragma unroll
      for (int j = 0; j < V / 2; ++j) {
        if (j < half) {
          const float send = up ? v[j] : v[j + half];
          const float keep = up ? v[j + half] : v[j];
          v[j] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
        }
      }
      count = half;
    } else {
      v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], o);
    }
  }
  return v[0];
}

template <typename T, int D>
__global__ __launch_bounds__(NT_ANCH, 7) void anchors_kernel(const T *__restrict__ K, int Tn,
                                                          int blk, int n_blocks, int window,
                                                          float *__restrict__ esum,
                                                          float *__restrict__ a) {
  using R = GroupRow<T, D>;
  constexpr int P2 = R::P2;
  // [NSTREAM][window + NB]: 1/|k| of row j at slot j % (window + NB).  A batch
  // writes NB distinct slots and never one that it reads (rows i - window < i0
  // sit at least window + 1 rows back), so no two lanes touch a slot in the same
  // batch.
  extern __shared__ float ring_all[];
  __shared__ __align__(16) float sums[NSTREAM][D];  // a stream's sum of kh over [c0, e), then [s, e)
  __shared__ __align__(16) float sils[NSTREAM][D];  // a stream's sum of kh over [c0, s)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane & (GW - 1);     // lane within the stream's group
  const int gbase = lane & ~(GW - 1);  // the group's first lane
  const int sid = warp * NSW + lane / GW;
  const long unit = blockIdx.x / n_blocks;
  const int bj = blockIdx.x % n_blocks;
  const int lo = min(Tn, bj * blk), hi = min(Tn, lo + blk);
  const T *Ku = K + unit * (long)Tn * D;
  const int RW = window + NB;
  float *ring = ring_all + sid * RW;
  float *ac = a + (unit * 3 + 2) * (long)Tn;
  const uint64_t keep_pol = tc::make_policy_evict_last();   // read again `window` rows later
  const uint64_t last_pol = tc::make_policy_evict_first();  // last read

  // The stream's tokens [s, e): spans are whole windows, so every stream of the
  // CTA has the same phase against the window-aligned chunks and the streams
  // of a warp take the same branches batch by batch.
  const int span = ((hi - lo + NSTREAM - 1) / NSTREAM + window - 1) / window * window;
  const int s = min(hi, lo + sid * span), e = min(hi, s + span);
  const bool live = s < e;
  // this lane's pairs of the stream's sums (kept in shared memory: they change
  // once a chunk)
  auto tot = [&](int p) -> float2 & { return *reinterpret_cast<float2 *>(&sums[sid][R::feature(g, p)]); };
  auto sil = [&](int p) -> float2 & { return *reinterpret_cast<float2 *>(&sils[sid][R::feature(g, p)]); };
#pragma unroll
  for (int p = 0; p < P2; ++p) sil(p) = make_float2(0.f, 0.f);

  const int c0 = (s / window) * window;  // the chunk start the stream walks from
  float2 P[P2], Q[P2];
#pragma unroll
  for (int p = 0; p < P2; ++p) P[p] = Q[p] = make_float2(0.f, 0.f);
  // warm-up: the full chunk before c0 (its total starts Q; its 1/|k| fill the ring)
  {
    const bool warm = live && c0 > 0;
    for (int k0 = 0; k0 < window; k0 += NB) {
      const int i0 = c0 - window + k0;
      float2 x[NB][P2];
      float ss[NB];
#pragma unroll
      for (int t = 0; t < NB; ++t) {
        const bool use = warm && k0 + t < window;
        R::load(Ku + (long)(use ? i0 + t : 0) * D, g, keep_pol, x[t]);
        float2 q2 = __fmul2_rn(x[t][0], x[t][0]);
#pragma unroll
        for (int p = 1; p < P2; ++p) q2 = __ffma2_rn(x[t][p], x[t][p], q2);
        ss[t] = use ? hsum(q2) : 0.f;
      }
      const float tt = reduce_scatter_group<NB>(ss, g);  // group lanes OWN t ..: token t
      const float my_inv = tt > 0.f ? rsqrtf(tt) : 0.f;
      const int mt = g / OWN;
      if (warm && g % OWN == 0 && k0 + mt < window) ring[(i0 + mt) % RW] = my_inv;
#pragma unroll
      for (int t = 0; t < NB; ++t) {
        const float inv = __shfl_sync(0xFFFFFFFFu, my_inv, gbase + OWN * t);
        if (warm && k0 + t < window) {
          const float2 inv2 = make_float2(inv, inv);
#pragma unroll
          for (int p = 0; p < P2; ++p) P[p] = __ffma2_rn(x[t][p], inv2, P[p]);
        }
      }
    }
  }
  // the first chunk reset moves the warm-up total into Q; keep it out of `tot`
#pragma unroll
  for (int p = 0; p < P2; ++p) tot(p) = make_float2(-P[p].x, -P[p].y);
  __syncwarp();
  int r = 0;         // i - (chunk start), i.e. i % window, kept as a running counter
  int rs = c0 % RW;  // i0 % RW
  // One batch of NB tokens of every stream of the warp.  FAST (taken only when
  // it holds for both streams): the batch lies inside [s, e), its leaving rows
  // are real rows (i0 >= window) and window % NB == 0, so no token needs a
  // bounds check and a chunk can only start at the batch's first token.
  // x: this batch's new rows; xn: the next batch's, in flight during this batch.
  // Rows past e or before 0 load an in-range row instead (no branch): a token
  // past e is never used.
  float2 x[NB][P2], xn[NB][P2], y[NB][P2], yn[NB][P2];
  auto load_next = [&](const int i0) {
#pragma unroll
    for (int t = 0; t < NB; ++t) {
      const int i = max(0, min(i0 + t, e - 1));
      R::load(Ku + (long)i * D, g, keep_pol, xn[t]);
      // the leaving row (a row before 0 loads row 0 instead and is scaled by 0)
      R::load(Ku + (long)max(i - window, 0) * D, g, last_pol, yn[t]);
    }
  };
  auto batch = [&](const int i0, auto fast_tag) {
    constexpr bool FAST = decltype(fast_tag)::value;
    float ss[NB];
#pragma unroll
    for (int t = 0; t < NB; ++t) {
      float2 q2 = __fmul2_rn(x[t][0], x[t][0]);
#pragma unroll
      for (int p = 1; p < P2; ++p) q2 = __ffma2_rn(x[t][p], x[t][p], q2);
      ss[t] = hsum(q2);
    }
    const float tt = reduce_scatter_group<NB>(ss, g);
    // group lanes OWN t .. own token t: swap its 1/|k| into the ring, take out the leaving row's
    const float my_inv = tt > 0.f ? rsqrtf(tt) : 0.f;
    float my_old = 0.f;
    {
      // slot of row j is j % RW; rs tracks i0 % RW, and (i - window) % RW is
      // (i + NB) % RW because RW = window + NB
      const int mt = g / OWN, i = i0 + mt;
      int sn = rs + mt;
      if (sn >= RW) sn -= RW;
      int so = sn + NB;
      if (so >= RW) so -= RW;
      if (g % OWN == 0 && (FAST || i < e)) {
        if (FAST || (i >= window && i - window < i0)) my_old = ring[so];
        ring[sn] = my_inv;
      }
    }
    rs += NB;
    if (rs >= RW) rs -= RW;
    float part[2 * NB];
#pragma unroll
    for (int t = 0; t < NB; ++t) {
      const int i = i0 + t;
      const float inv = __shfl_sync(0xFFFFFFFFu, my_inv, gbase + OWN * t);
      float old = __shfl_sync(0xFFFFFFFFu, my_old, gbase + OWN * t);
      if constexpr (!FAST) {
        if (window < NB) {  // the leaving row may be in this very batch
          const float same = __shfl_sync(0xFFFFFFFFu, my_inv, gbase + OWN * max(t - window, 0));
          if (t >= window) old = same;
        }
      }
      float dot = 0.f, nrm = 0.f;
      if (FAST || i < e) {
        if ((!FAST || t == 0) && r == 0) {  // a new chunk: the previous total becomes Q
#pragma unroll
          for (int p = 0; p < P2; ++p) {
            tot(p) = __fadd2_rn(tot(p), P[p]);
            Q[p] = P[p];
            P[p] = make_float2(0.f, 0.f);
          }
        }
        const float2 inv2 = make_float2(inv, inv), nold2 = make_float2(-old, -old);
        float2 d2 = make_float2(0.f, 0.f), n2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < P2; ++p) {
          P[p] = __ffma2_rn(x[t][p], inv2, P[p]);
          Q[p] = __ffma2_rn(y[t][p], nold2, Q[p]);
          const float2 w = __fadd2_rn(P[p], Q[p]);
          d2 = __ffma2_rn(x[t][p], w, d2);
          n2 = __ffma2_rn(w, w, n2);
        }
        dot = hsum(d2);
        nrm = hsum(n2);
        if constexpr (!FAST) {
          if (i == s - 1) {
#pragma unroll
            for (int p = 0; p < P2; ++p) sil(p) = P[p];
          }
          r = (r + 1 == window) ? 0 : r + 1;
        }
      }
      part[2 * t] = dot;
      part[2 * t + 1] = nrm;
    }
    if constexpr (FAST) {
      r += NB;
      if (r == window) r = 0;
    }
    const float v = reduce_scatter_group<2 * NB>(part, g);
    // group lane OWN t holds token t's <k, window sum> (and 1/|k|); lane OWN t + OWN/2
    // the window's |.|^2
    const float nrm = __shfl_down_sync(0xFFFFFFFFu, v, OWN / 2);
    if (g % OWN == 0) {
      const int i = i0 + g / OWN;
      // cos(kh_i, window sum) with |kh_i| = 1 (a zero key has dot 0)
      if (FAST || (i >= s && i < e)) ac[i] = nrm > 0.f ? -(v * my_inv) * rsqrtf(nrm) : 0.f;
    }
    __syncwarp();  // this batch's ring writes before the next batch's reads
  };
  const bool can_fast = window % NB == 0;
  load_next(c0);
  for (int i0 = c0; __any_sync(0xFFFFFFFFu, live && i0 < e); i0 += NB) {
#pragma unroll
    for (int t = 0; t < NB; ++t)
#pragma unroll
      for (int p = 0; p < P2; ++p) {
        x[t][p] = xn[t][p];
        y[t][p] = yn[t][p];
      }
    load_next(i0 + NB);
    if (__all_sync(0xFFFFFFFFu, can_fast && live && i0 >= s && i0 >= window && i0 + NB <= e))
      batch(i0, std::integral_constant<bool, true>());
    else
      batch(i0, std::integral_constant<bool, false>());
  }
  if (live) {
#pragma unroll
    for (int p = 0; p < P2; ++p)
      tot(p) = __fadd2_rn(__fadd2_rn(tot(p), P[p]), make_float2(-sil(p).x, -sil(p).y));
  } else {
#pragma unroll
    for (int p = 0; p < P2; ++p) tot(p) = make_float2(0.f, 0.f);
  }
  // block sum of kh over the streams
  __syncthreads();
  for (int f = threadIdx.x; f < D; f += NT_ANCH) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NSTREAM; ++w) t += sums[w][f];
    esum[(unit * n_blocks + bj) * (long)D + f] = t;
  }
}

// ---- 2. stable and episodic anchors ----------------------------------------------
// Four lanes per key: lane q of a group reads the 16-byte pieces q, q+4, q+8, ...
// of its key (each load of the group covers whole 32-byte sectors of one row),
// reads the matching slices of S and E from shared memory (the four lanes of a
// group read four different addresses, every group the same: no conflicts),
// and the group adds its four partial <k, S>, <k, E> and |k|^2 with two
// shuffles.  A
// warp takes 8 keys a step; the next two steps' loads are in flight during
// this step's arithmetic.
template <typename T, int D>
__global__ __launch_bounds__(NT_SCAN) void global_kernel(const T *__restrict__ K, int Tn, int blk,
                                                         int n_blocks,
                                                         const float *__restrict__ esum,
                                                         float *__restrict__ a) {
  constexpr int NC = D * (int)sizeof(T) / 64;  // 16-byte pieces per lane
  constexpr int FC = 16 / (int)sizeof(T);      // features per piece
  constexpr int FS = 64 / (int)sizeof(T);      // feature stride between a lane's pieces
  __shared__ __align__(16) float S[D], E[D];
  __shared__ float nrm[2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int q = lane & 3, g = lane >> 2;
  const long unit = blockIdx.x / n_blocks;
  const int bj = blockIdx.x % n_blocks;
  const int lo = min(Tn, bj * blk), hi = min(Tn, lo + blk);
  const float *eu = esum + unit * (long)n_blocks * D;
  for (int f = threadIdx.x; f < D; f += NT_SCAN) {
    float t = 0.f;
    for (int j = 0; j < n_blocks; ++j) t += eu[(long)j * D + f];
    S[f] = t;
    E[f] = eu[(long)bj * D + f];
  }
  __syncthreads();
  if (warp == 0) {  // anchor norms
    float ns = 0.f, ne = 0.f;
    for (int f = lane; f < D; f += 32) {
      ns = fmaf(S[f], S[f], ns);
      ne = fmaf(E[f], E[f], ne);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ns += __shfl_xor_sync(0xFFFFFFFFu, ns, o);
      ne += __shfl_xor_sync(0xFFFFFFFFu, ne, o);
    }
    if (lane == 0) {
      nrm[0] = ns > 0.f ? rsqrtf(ns) : 0.f;
      nrm[1] = ne > 0.f ? rsqrtf(ne) : 0.f;
    }
  }
  __syncthreads();
  const float rS = nrm[0], rE = nrm[1];
  const char *Ku = reinterpret_cast<const char *>(K + unit * (long)Tn * D);
  float *as = a + (unit * 3 + 0) * (long)Tn;
  float *ae = a + (unit * 3 + 1) * (long)Tn;
  auto load = [&](int t0, uint4 (&w)[NC]) {
    const uint4 *row = reinterpret_cast<const uint4 *>(Ku + (long)min(t0 + g, hi - 1) * (D * (int)sizeof(T)));
#pragma unroll
    for (int c = 0; c < NC; ++c) w[c] = __ldg(row + 4 * c + q);
  };
  const int step = 8 * NWARP;
  int t0 = lo + 8 * warp;
  uint4 wn[NC], wnn[NC];  // the next two steps' pieces, in flight
  if (t0 < hi) load(t0, wn);
  if (t0 + step < hi) load(t0 + step, wnn);
  for (; t0 < hi; t0 += step) {
    uint4 w[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      w[c] = wn[c];
      wn[c] = wnn[c];
    }
    if (t0 + 2 * step < hi) load(t0 + 2 * step, wnn);
    float2 ds = make_float2(0.f, 0.f), de = ds, nk = ds;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const uint32_t u[4] = {w[c].x, w[c].y, w[c].z, w[c].w};
      // this lane's features of piece c, and the anchors' values for them
      const float2 *sv = reinterpret_cast<const float2 *>(S + c * FS + q * FC);
      const float2 *ev = reinterpret_cast<const float2 *>(E + c * FS + q * FC);
#pragma unroll
      for (int e = 0; e < FC / 2; ++e) {
        float2 x;
        if constexpr (sizeof(T) == 2)  // bf16: a word holds two features
          x = make_float2(__uint_as_float(u[e] << 16), __uint_as_float(u[e] & 0xFFFF0000u));
        else
          x = make_float2(__uint_as_float(u[2 * e]), __uint_as_float(u[2 * e + 1]));
        ds = __ffma2_rn(x, sv[e], ds);
        de = __ffma2_rn(x, ev[e], de);
        nk = __ffma2_rn(x, x, nk);
      }
    }
    float v0 = hsum(ds), v1 = hsum(de), v2 = hsum(nk);
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, o);
      v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, o);
      v2 += __shfl_xor_sync(0xFFFFFFFFu, v2, o);
    }
    const int i = t0 + g;
    if (q == 0 && i < hi) {
      const float rk = v2 > 0.f ? rsqrtf(v2) : 0.f;
      as[i] = -(v0 * rk) * rS;
      ae[i] = -(v1 * rk) * rE;
    }
  }
}

// ---- 3. discriminative power per (unit, scale) -----------------------------------
// Calls f(x) for every value of v[0..n) with 16-byte loads (scalars up to the first
// 16-byte boundary and after the last), four vectors in flight per thread.
template <typename F>
__device__ __forceinline__ void for_values(const float *__restrict__ v, int n, F &&f) {
  const int mis = (int)((reinterpret_cast<uintptr_t>(v) >> 2) & 3);
  const int pre = min(n, (4 - mis) & 3), n4 = (n - pre) >> 2, tail = pre + 4 * n4;
  const float4 *v4 = reinterpret_cast<const float4 *>(v + pre);
  for (int base = threadIdx.x; base < n4; base += 4 * NT_DISC) {
    float4 q[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = base + u * NT_DISC;
      q[u] = j < n4 ? __ldg(v4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (base + u * NT_DISC < n4) {
        f(q[u].x);
        f(q[u].y);
        f(q[u].z);
        f(q[u].w);
      }
  }
  const int t = threadIdx.x;
  if (t < pre) f(__ldg(v + t));
  else if (t < pre + (n - tail)) f(__ldg(v + tail + (t - pre)));
}

// D = (sum of the m largest of v) / m - (sum of the m smallest) / m.  Both radix
// selects (order-preserving keys for the largest, their complements for the
// smallest) share every pass over v: 4 histogram passes of 8 bits and one sum
// pass.  Each sum is the values strictly beyond the boundary key plus the right
// number of copies of the boundary value; block reductions in a fixed order.
__global__ __launch_bounds__(NT_DISC, 1) void disc_kernel(const float *__restrict__ a, int Tn,
                                                          int m, float *__restrict__ D) {
  constexpr int NW = NT_DISC / 32;
  extern __shared__ uint32_t hist[];  // [2][NW][256]
  __shared__ uint32_t tot[2][256];
  __shared__ uint32_t sh_prefix[2];
  __shared__ int sh_need[2];
  __shared__ float sh_b[2], red[2][NW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float *v = a + (long)blockIdx.x * Tn;  // blockIdx.x = unit * 3 + scale
  uint32_t prefix[2] = {0u, 0u}, mask = 0u;
  int need[2] = {m, m};
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < 2 * NW * 256; i += NT_DISC) hist[i] = 0u;
    __syncthreads();
    uint32_t *h0 = hist + warp * 256, *h1 = hist + (NW + warp) * 256;
    if (pass == 0) {
      // the complements' top byte is 255 minus the keys': one histogram serves both
      for_values(v, Tn, [&](float x) { atomicAdd(h0 + (order_key(x) >> 24), 1u); });
    } else {
      for_values(v, Tn, [&](float x) {
        const uint32_t u = order_key(x), ub = ~u;
        if ((u & mask) == prefix[0]) atomicAdd(h0 + ((u >> shift) & 255u), 1u);
        if ((ub & mask) == prefix[1]) atomicAdd(h1 + ((ub >> shift) & 255u), 1u);
      });
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 512; i += NT_DISC) {
      const int k = i >> 8, d = i & 255;
      uint32_t t = 0;
      if (pass == 0)
        for (int w = 0; w < NW; ++w) t += hist[w * 256 + (k ? 255 - d : d)];
      else
        for (int w = 0; w < NW; ++w) t += hist[(k * NW + w) * 256 + d];
      tot[k][d] = t;
    }
    __syncthreads();
    if (warp < 2) {  // warp 0 decides for the largest, warp 1 for the smallest
      const int k = warp;
      uint32_t mine = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) mine += tot[k][255 - 8 * lane - i];
      uint32_t incl = mine;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += y;
      }
      uint32_t above = incl - mine;
      if (above < (uint32_t)need[k] && (uint32_t)need[k] <= incl) {
        for (int i = 0; i < 8; ++i) {
          const int dgt = 255 - 8 * lane - i;
          if ((uint32_t)need[k] <= above + tot[k][dgt]) {
            sh_prefix[k] = prefix[k] | ((uint32_t)dgt << shift);
            sh_need[k] = need[k] - (int)above;
            break;
          }
          above += tot[k][dgt];
        }
      }
    }
    __syncthreads();
    prefix[0] = sh_prefix[0];
    prefix[1] = sh_prefix[1];
    need[0] = sh_need[0];
    need[1] = sh_need[1];
    mask |= 255u << shift;
    __syncthreads();
  }
  float ptop = 0.f, pbot = 0.f;
  for_values(v, Tn, [&](float x) {
    const uint32_t u = order_key(x), ub = ~u;
    if (u > prefix[0]) ptop += x;
    if (u == prefix[0]) sh_b[0] = x;  // every value with the boundary key is equal (up to the sign of 0)
    if (ub > prefix[1]) pbot += x;
    if (ub == prefix[1]) sh_b[1] = x;
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ptop += __shfl_xor_sync(0xFFFFFFFFu, ptop, o);
    pbot += __shfl_xor_sync(0xFFFFFFFFu, pbot, o);
  }
  if (lane == 0) {
    red[0][warp] = ptop;
    red[1][warp] = pbot;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float top = 0.f, bot = 0.f;
    for (int w = 0; w < NW; ++w) {
      top += red[0][w];
      bot += red[1][w];
    }
    top += (float)need[0] * sh_b[0];
    bot += (float)need[1] * sh_b[1];
    D[blockIdx.x] = (top - bot) / (float)m;
  }
}

// ---- 4. weights, surprise, routing ------------------------------------------------
__global__ void final_kernel(const float *__restrict__ a, const float *__restrict__ D, int Tn,
                             long units, float lp0, float lp1, float lp2, float thresh,
                             float *__restrict__ score, float *__restrict__ w_out) {
  for (long u = blockIdx.y; u < units; u += gridDim.y) {
    const float z0 = D[u * 3 + 0] + lp0, z1 = D[u * 3 + 1] + lp1, z2 = D[u * 3 + 2] + lp2;
    const float zm = fmaxf(z0, fmaxf(z1, z2));
    const float e0 = expf(z0 - zm), e1 = expf(z1 - zm), e2 = expf(z2 - zm);
    const float es = e0 + e1 + e2;
    const float w0 = e0 / es, w1 = e1 / es, w2 = e2 / es;
    if (w_out && blockIdx.x == 0 && threadIdx.x == 0) {
      w_out[u * 3 + 0] = w0;
      w_out[u * 3 + 1] = w1;
      w_out[u * 3 + 2] = w2;
    }
    const float *as = a + (u * 3 + 0) * (long)Tn;
    const float *ae = as + Tn;
    const float *ac = ae + Tn;
    float *su = score + u * (long)Tn;
    auto route = [&](float x0, float x1, float x2) {
      const float mean = (x0 + x1 + x2) / 3.f;
      const float var = ((x0 - mean) * (x0 - mean) + (x1 - mean) * (x1 - mean) +
                         (x2 - mean) * (x2 - mean)) / 3.f;
      const float sig = sqrtf(var);
      return sig > thresh ? fmaxf(x0, fmaxf(x1, x2)) : w0 * x0 + w1 * x1 + w2 * x2;
    };
    const int stride = gridDim.x * blockDim.x;
    int i0 = 0;  // tokens from here on take the scalar loop
    if (((reinterpret_cast<uintptr_t>(as) | reinterpret_cast<uintptr_t>(ae) |
          reinterpret_cast<uintptr_t>(ac) | reinterpret_cast<uintptr_t>(su)) & 15) == 0) {
      // 16-byte vectors of four tokens, two a thread in flight
      const int n4 = Tn >> 2;
      const float4 *as4 = reinterpret_cast<const float4 *>(as), *ae4 = reinterpret_cast<const float4 *>(ae),
                   *ac4 = reinterpret_cast<const float4 *>(ac);
      float4 *su4 = reinterpret_cast<float4 *>(su);
      for (int q0 = blockIdx.x * blockDim.x + threadIdx.x; q0 < n4; q0 += 2 * stride) {
        float4 x0[2], x1[2], x2[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int q = min(q0 + h * stride, n4 - 1);
          x0[h] = __ldg(as4 + q);
          x1[h] = __ldg(ae4 + q);
          x2[h] = __ldg(ac4 + q);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int q = q0 + h * stride;
          if (q < n4)
            su4[q] = make_float4(route(x0[h].x, x1[h].x, x2[h].x), route(x0[h].y, x1[h].y, x2[h].y),
                                 route(x0[h].z, x1[h].z, x2[h].z), route(x0[h].w, x1[h].w, x2[h].w));
        }
      }
      i0 = 4 * n4;
    }
    for (int i = i0 + blockIdx.x * blockDim.x + threadIdx.x; i < Tn; i += stride)
      su[i] = route(as[i], ae[i], ac[i]);
  }
}

template <typename T, int D>
int run_nested(const void *K, long units, int Tn, int window, int n_blocks, int n_disc,
               float lp0, float lp1, float lp2, float thresh, float *score, float *w_out,
               float *a, void *ws, cudaStream_t st) {
  const int blk = (Tn + n_blocks - 1) / n_blocks;
  float *esum = static_cast<float *>(ws);
  float *Dw = esum + units * (long)n_blocks * D;
  const unsigned grid = (unsigned)(units * n_blocks);
  const size_t ring = (size_t)NSTREAM * (window + 4) * sizeof(float);
  if (ensure_smem((const void *)anchors_kernel<T, D>, ring))
    return cuda_failure(cudaErrorInvalidValue, "nested anchors kernel: shared memory");
  anchors_kernel<T, D><<<grid, NT_ANCH, ring, st>>>(static_cast<const T *>(K), Tn, blk, n_blocks,
                                                    window, esum, a);
  int rc = launch_status();
  if (rc) return rc;
  global_kernel<T, D><<<grid, NT_SCAN, 0, st>>>(static_cast<const T *>(K), Tn, blk, n_blocks,
                                                esum, a);
  if ((rc = launch_status())) return rc;
  const size_t dsm = (size_t)2 * (NT_DISC / 32) * 256 * sizeof(uint32_t);
  if (ensure_smem((const void *)disc_kernel, dsm))
    return cuda_failure(cudaErrorInvalidValue, "nested disc kernel: shared memory");
  disc_kernel<<<(unsigned)(units * 3), NT_DISC, dsm, st>>>(a, Tn, n_disc, Dw);
  if ((rc = launch_status())) return rc;
  const dim3 fgrid((unsigned)min((Tn + 1023) / 1024, 64), (unsigned)min(units, 65535L));
  final_kernel<<<fgrid, 256, 0, st>>>(a, Dw, Tn, units, lp0, lp1, lp2, thresh, score, w_out);
  return launch_status();
}

}  // namespace

size_t nested_workspace_bytes(long units, int T, int d, int n_blocks, bool with_a) {
  size_t b = (size_t)units * n_blocks * d * sizeof(float) + (size_t)units * 4 * sizeof(float);
  b = (b + 255) & ~(size_t)255;
  if (with_a) b += (size_t)units * 3 * T * sizeof(float);
  return b;
}

int launch_score_nested(const void *K, int B, int H, int T, int d, int dtype, int window,
                        int n_blocks, int n_disc, float lp0, float lp1, float lp2, float thresh,
                        float *score, float *w_out, float *a_out, void *ws, cudaStream_t st) {
  const long units = (long)B * H;
  float *a = a_out;
  if (!a) {
    const size_t off = nested_workspace_bytes(units, T, d, n_blocks, false);
    a = reinterpret_cast<float *>(static_cast<char *>(ws) + off);
  }
  if (dtype == KV_BF16) {
    if (d == 128)
      return run_nested<__nv_bfloat16, 128>(K, units, T, window, n_blocks, n_disc, lp0, lp1, lp2,
                                            thresh, score, w_out, a, ws, st);
    return run_nested<__nv_bfloat16, 64>(K, units, T, window, n_blocks, n_disc, lp0, lp1, lp2,
                                         thresh, score, w_out, a, ws, st);
  }
  if (d == 128)
    return run_nested<float, 128>(K, units, T, window, n_blocks, n_disc, lp0, lp1, lp2, thresh,
                                  score, w_out, a, ws, st);
  return run_nested<float, 64>(K, units, T, window, n_blocks, n_disc, lp0, lp1, lp2, thresh, score,
                               w_out, a, ws, st);
}

}  // namespace kvc
