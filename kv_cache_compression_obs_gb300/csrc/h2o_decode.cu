// h2o_decode.cu -- one H2O decode step over a preallocated slot cache.
//
// H2O page: 问题形式化 (|S_i| = k, at most one eviction per step, attention
// renormalised over the kept keys), 贪心驱逐算法 (Algorithm 1: accumulate the
// softmax into a per-token score, evict the lowest), 双缓冲 (the recent window
// is protected), FlexGen 改造 (the evicted slot is overwritten in place; the
// score vector is updated as a by-product of the attention kernel).
//
// A unit is (b, KV head); its attended rows are the filled slots 0..n-1 plus the
// new token (row n).  Two launches per step:
//
//   stream   -- persistent, one CTA per SM.  Every unit is cut into blocks of RB
//               rows, the blocks of all units are laid end to end and each CTA
//               takes one contiguous range of them.  A producer warp streams each
//               block's K rows and V rows into two rings of shared-memory stages
//               with bulk copies (exactly the cached rows, L2 evict-first); all
//               consumer warps share every block, RB / NCW rows each, so that a
//               stage is held only briefly and most of the rings are in flight.
//               K stage: 8 lanes per row (q of the lane's eighth of d in
//               registers, a butterfly across the 8 lanes), logits in log2 units
//               l_gj = scale log2(e) <q_g, k_j> for the G query heads of the
//               group, also written to the workspace.  Weights 2^(l_gj - r_g)
//               against a per-warp reference r_g that moves (rescaling the warp's
//               sums) only when a block's max passes it by more than kLazyLog2.
//               V stage: one row at a time across the lanes, o_g += w_gj v_j.
//               When the CTA's part of a unit is done, its warps' (r, Z, o) are
//               combined into one partial per (unit, CTA).
//   finalize -- CE CTAs per unit: combine the partials into o_out; turn the
//               stored logits into probabilities P_j = sum_g 2^(l_gj - (M_g +
//               log2 Z_g)), add them to the slots' accumulators and take each
//               CTA's (acc, pos)-smallest slot outside the recent window and
//               outside the first `sink` positions (attention sinks).  Each
//               CTA publishes its candidate and counts itself in on the unit's
//               arrival counter (zeroed by the stream kernel); the last to
//               arrive picks the smallest (and the new token itself when
//               recent == 0) and appends the new token or writes it over the
//               victim.  No CTA waits for another.  Every load that does not
//               depend on the unit's length (its partials, the CTA's slots,
//               shared out by capacity) is issued before the length arrives.
//
// Workspace: logits [units][G][cap+1] and the per-(unit, CTA) partials (m, Z)
// [units][PM][G] and o [units][PM][G][D], all float.
#include <cmath>
#include <type_traits>

#include "kvc_internal.cuh"
#include "tc_common.cuh"

namespace kvc {
namespace {

constexpr int RB_MIN = 64;   // rows per block of the widest rows (bounds the partials per unit)
constexpr int NCW = 8;       // consumer warps: every block is shared by all of them
constexpr int LPR = 8;       // lanes per row in the K stage
constexpr int RPI = 32 / LPR;  // rows per K step of a warp
constexpr float kLazyLog2 = 16.f;  // the weights' reference moves only when passed by more (log2 units)
constexpr int PER_MIN = 8;   // a CTA takes at least this many blocks (bounds partials per unit)
constexpr int kSmemBudget = 220 * 1024;
constexpr int kMaxStages = 16;
constexpr long long kWaitBudget = 2000000000LL;  // clock cycles (~1 s) before a wait gives up
constexpr long long kDrainBudget = 200000000LL;  // ~0.1 s for copies in flight at exit
constexpr int BAR_CONS = 1;  // named barrier of the consumer warps
constexpr int NTF = 128;     // finalize threads per CTA: small enough (with its registers) to
                             // share an SM with a stream CTA of the other half of the rows
constexpr int CE = 4;        // finalize CTAs per unit
constexpr int RU = 8;        // finalize slots per thread in flight

__device__ __forceinline__ bool better(float a, int p, float ba, int bp) {
  return a < ba || (a == ba && p < bp);
}

// Shared-memory layout of the stream kernel for element type T, head dim D and
// group size G.  Stages hold whole rows, contiguous as in global memory.
template <typename T, int D, int G>
struct DGeo {
  static constexpr int ROWB = D * (int)sizeof(T);  // bytes per K or V row
  static constexpr int RB = ROWB <= 256 ? 128 : RB_MIN;  // rows per block
  static constexpr int RPW = RB / NCW;             // rows of a block per consumer warp
  static constexpr int KIT = RPW / RPI;            // K steps per block
  static constexpr int STAGE = RB * ROWB;          // one block of K (or V) rows
  static constexpr int CPL = ROWB / 16 / LPR;      // 16-byte chunks per lane of a K row
  static constexpr int HG = G < 4 ? G : 4;         // query heads per K pass
  static constexpr int NPASS = G / HG;
  static constexpr int PBW = G * D + 2 * G;        // one warp's partial: o[G][D], m[G], Z[G]
  static constexpr int QS_BYTES = G * D * 4;       // q of the unit, fp32
  static constexpr int PW_BYTES = NCW * RPW * G * 4;  // per-warp weights exp(l - m) of its rows
  static constexpr int PB_BYTES = NCW * PBW * 4;
  static constexpr int SC_BYTES = NCW * G * 4;     // combine scales
  static constexpr int MISC_BYTES = 1024;          // barriers, flags
  static constexpr int FIXED = QS_BYTES + PW_BYTES + PB_BYTES + SC_BYTES + MISC_BYTES;
  static constexpr int S_FIT = (kSmemBudget - 1024 - FIXED) / (2 * STAGE);
  static constexpr int S = S_FIT > kMaxStages ? kMaxStages : S_FIT;  // depth of each ring
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = S * STAGE;
  static constexpr int QS_OFF = 2 * S * STAGE;
  static constexpr int PW_OFF = QS_OFF + QS_BYTES;
  static constexpr int PB_OFF = PW_OFF + PW_BYTES;
  static constexpr int SC_OFF = PB_OFF + PB_BYTES;
  static constexpr int MISC_OFF = SC_OFF + SC_BYTES;
  static constexpr int SMEM = 1024 /*alignment slack*/ + MISC_OFF + MISC_BYTES;
  static_assert(ROWB % (16 * LPR) == 0 && CPL >= 1, "a K row splits evenly over its lanes");
  static_assert(G % HG == 0, "whole head passes");
  static_assert(RPW % RPI == 0 && RPW % 8 == 0, "whole K steps and V batches");
  static_assert(S >= 2, "ring depth");
  static_assert(4 * kMaxStages * 8 + 64 + 8 * G <= MISC_BYTES, "misc area");
};

struct Cand {
  float acc;
  int pos;
  int slot;       // -2: no candidate
  float accself;  // the new token's score
};

struct Ws {      // workspace carve-up
  float *lgw;    // [units][G][cap+1] logits
  float2 *pmz;   // [units][PM][G] per-(unit, CTA) max and normaliser
  float *po;     // [units][PM][G][D] per-(unit, CTA) output shares (relative to the max)
  Cand *cnd;     // [units][CE] the finalize CTAs' eviction candidates
  int *cnt;      // [units] finalize arrivals (zeroed by the stream kernel of the same step)
};

inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }
__host__ __device__ inline int blocks_per_unit(int cap, int rb) { return (cap + 1 + rb - 1) / rb; }
// Partials per unit: a unit's NB blocks meet at most ceil(NB / per) + 1 CTA
// ranges, and every range holds at least PER_MIN blocks unless one CTA runs
// alone; blocks are never shorter than RB_MIN rows.
__host__ __device__ inline int partials_per_unit(int cap) {
  return (blocks_per_unit(cap, RB_MIN) + PER_MIN - 1) / PER_MIN + 1;
}

Ws carve(void *ws, long units, int G, int cap, int d) {
  const int PM = partials_per_unit(cap);
  Ws w;
  char *p = static_cast<char *>(ws);
  w.lgw = reinterpret_cast<float *>(p);
  p += align256((size_t)units * G * (cap + 1) * 4);
  w.pmz = reinterpret_cast<float2 *>(p);
  p += align256((size_t)units * PM * G * 8);
  w.po = reinterpret_cast<float *>(p);
  p += align256((size_t)units * PM * G * d * 4);
  w.cnd = reinterpret_cast<Cand *>(p);
  p += align256((size_t)units * CE * sizeof(Cand));
  w.cnt = reinterpret_cast<int *>(p);
  return w;
}

// EV consecutive elements of a row (EV * sizeof(T) = 4, 8 or 16 bytes).
template <typename T, int EV>
struct RowPiece {
  static constexpr int BYTES = EV * (int)sizeof(T);
  using Word = typename std::conditional<BYTES == 16, uint4,
               typename std::conditional<BYTES == 8, uint2, uint32_t>::type>::type;
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

// The CTAs of the stream kernel whose block ranges meet unit u: the first, and how many.
struct Span {
  int first, count;
};
__device__ __forceinline__ Span unit_span(long u, int NB, long per) {
  const int first = static_cast<int>((u * NB) / per);
  const int last = static_cast<int>(((u + 1) * NB - 1) / per);
  return Span{first, last - first + 1};
}

__device__ __forceinline__ void fail(volatile int *abort_flag, int *status) {
  *abort_flag = 1;
  if (status) atomicExch(status, (int)KV_ERR_TIMEOUT);
}

// sum over the LPR = 8 lanes of a row of the HG values v[] (lanes 8r .. 8r+7):
// after the butterfly, lane pp holds the total of value pp / (8 / HG).
template <int HG>
__device__ __forceinline__ float row_butterfly(float (&v)[HG], int pp) {
  if constexpr (HG == 4) {
    const bool up4 = pp & 4;
    float a0 = up4 ? v[2] : v[0], a1 = up4 ? v[3] : v[1];
    const float s0 = up4 ? v[0] : v[2], s1 = up4 ? v[1] : v[3];
    a0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 4);
    a1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 4);
    const bool up2 = pp & 2;
    float b = up2 ? a1 : a0;
    b += __shfl_xor_sync(0xFFFFFFFFu, up2 ? a0 : a1, 2);
    return b + __shfl_xor_sync(0xFFFFFFFFu, b, 1);
  } else if constexpr (HG == 2) {
    const bool up4 = pp & 4;
    float a = up4 ? v[1] : v[0];
    a += __shfl_xor_sync(0xFFFFFFFFu, up4 ? v[0] : v[1], 4);
    a += __shfl_xor_sync(0xFFFFFFFFu, a, 2);
    return a + __shfl_xor_sync(0xFFFFFFFFu, a, 1);
  } else {
    float a = v[0];
    a += __shfl_xor_sync(0xFFFFFFFFu, a, 4);
    a += __shfl_xor_sync(0xFFFFFFFFu, a, 2);
    return a + __shfl_xor_sync(0xFFFFFFFFu, a, 1);
  }
}

template <typename T, int D, int G>
__device__ __forceinline__ void decode_stream_body(
    const T *__restrict__ Kc, const T *__restrict__ Vc, const T *__restrict__ q,
    const T *__restrict__ k_new, const T *__restrict__ v_new, const int32_t *__restrict__ len, int Hq,
    int Hkv, int cap, float c_log2, int alg1, long total, long per, Ws ws, int *__restrict__ dev_status) {
  using Geo = DGeo<T, D, G>;
  constexpr int RB = Geo::RB;
  constexpr int RPW = Geo::RPW;
  constexpr int KIT = Geo::KIT;
  constexpr int S = Geo::S;
  constexpr int NCT = 32 * NCW;
  constexpr int EV = D / 32;  // V elements per lane
  constexpr int PBW = Geo::PBW;
  constexpr int EPL = Vec16<T>::N;
  constexpr int CPL = Geo::CPL;
  constexpr int HG = Geo::HG;
  constexpr int DUP = LPR / HG;  // lanes of a row holding the same head's logit
  using RP = RowPiece<T, EV>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char *sK = sm + Geo::K_OFF;
  unsigned char *sV = sm + Geo::V_OFF;
  float *qs = reinterpret_cast<float *>(sm + Geo::QS_OFF);
  float *pw = reinterpret_cast<float *>(sm + Geo::PW_OFF);
  float *pb = reinterpret_cast<float *>(sm + Geo::PB_OFF);
  float *sc = reinterpret_cast<float *>(sm + Geo::SC_OFF);
  uint64_t *kfull = reinterpret_cast<uint64_t *>(sm + Geo::MISC_OFF);
  uint64_t *kempty = kfull + kMaxStages;
  uint64_t *vfull = kempty + kMaxStages;
  uint64_t *vempty = vfull + kMaxStages;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(vempty + kMaxStages);
  float *fm = reinterpret_cast<float *>(sm + Geo::MISC_OFF + 4 * kMaxStages * 8 + 64);  // [G] max
  float *fz = fm + G;                                                                   // [G] normaliser

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NB = blocks_per_unit(cap, RB);
  const int PM = partials_per_unit(cap);
  const long lo = blockIdx.x * per;
  const long hi = min(total, lo + per);

  // the finalize kernel's arrival counters: each unit's by the CTA holding its first block
  for (long u = (lo + NB - 1) / NB + threadIdx.x; u * NB < hi; u += blockDim.x) ws.cnt[u] = 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(kfull + i, 1);
      tc::mbar_init(kempty + i, NCW);
      tc::mbar_init(vfull + i, 1);
      tc::mbar_init(vempty + i, NCW);
    }
    *abort_flag = 0;
    tc::mbar_fence_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------- producer (one lane) ----------------
    if (lane == 0 && lo < hi) {
      const uint64_t pol = tc::make_policy_evict_first();
      long cur_u = -1;
      int n = 0;
      long i = 0;
      for (long gb = lo; gb < hi; ++gb, ++i) {
        const long u = gb / NB;
        const int jb = static_cast<int>(gb % NB);
        if (u != cur_u) {
          cur_u = u;
          n = len[u];
          if (n < 0 || n > cap) n = 0;  // reported by the finalize kernel
        }
        const int rows = max(0, min(RB, n - jb * RB));  // cached rows in this block
        const uint32_t bytes = static_cast<uint32_t>(rows * Geo::ROWB);
        const long row0 = u * (long)cap + (long)jb * RB;
        const int si = static_cast<int>(i % S);
        const uint32_t ph = static_cast<uint32_t>((i / S) & 1);
        if (!tc::mbar_wait(kempty + si, ph ^ 1, kWaitBudget, abort_flag)) {
          fail(abort_flag, dev_status);
          break;
        }
        if (rows > 0) {
          tc::mbar_arrive_expect_tx(kfull + si, bytes);
          tc::bulk_load_hint(sK + si * Geo::STAGE, Kc + row0 * D, bytes, kfull + si, pol);
        } else {
          tc::mbar_arrive(kfull + si);
        }
        if (!tc::mbar_wait(vempty + si, ph ^ 1, kWaitBudget, abort_flag)) {
          ++i;  // this block's K copy may be in flight
          fail(abort_flag, dev_status);
          break;
        }
        if (rows > 0) {
          tc::mbar_arrive_expect_tx(vfull + si, bytes);
          tc::bulk_load_hint(sV + si * Geo::STAGE, Vc + row0 * D, bytes, vfull + si, pol);
        } else {
          tc::mbar_arrive(vfull + si);
        }
      }
      if (*abort_flag) {
        // copies still in flight land before the CTA may exit (bounded waits)
        for (long k = 1; k <= S && i - k >= 0; ++k) {
          const long ii = i - k;
          tc::mbar_wait(kfull + ii % S, (uint32_t)((ii / S) & 1), kDrainBudget, nullptr);
          tc::mbar_wait(vfull + ii % S, (uint32_t)((ii / S) & 1), kDrainBudget, nullptr);
        }
      }
    }
    __syncwarp();
    return;
  }

  // ---------------- consumers: warp w takes rows [RPW w, RPW w + RPW) of every block ----------------
  const int w = warp - 1;  // 0 .. NCW-1
  const int ct = threadIdx.x - 32;
  const int rs = lane / LPR;  // row of a K step
  const int pp = lane % LPR;  // this lane's part of that row
  const int hd = pp / DUP;    // head (within a pass) whose logit the lane ends with
  const bool writer = (pp % DUP) == 0;
  const int wr0 = RPW * w;    // this warp's first row of a block
  float *pww = pw + w * RPW * G;  // this warp's weights [RPW][G]
  bool ok = true;
  long i = 0;
  // A warp that gives up keeps walking the same items (without touching the
  // rings) so that every named barrier is reached by all consumer threads.
  for (long gb = lo; gb < hi;) {
    const long u = gb / NB;
    const long item_end = min(hi, (u + 1) * NB);
    const long b = u / Hkv;
    const int h = static_cast<int>(u % Hkv);
    int n = len[u];
    const bool valid = n >= 0 && n <= cap;
    if (!valid) n = 0;
    const int nc = valid ? n + (alg1 ? 0 : 1) : 0;  // attended rows
    const T *qg = q + (b * Hq + (long)h * G) * D;
    tc::named_bar_sync(BAR_CONS, NCT);  // the previous item's shared-memory readers are done
    for (int t = ct; t < G * D; t += NCT) qs[t] = to_f32(qg[t]);
    tc::named_bar_sync(BAR_CONS, NCT);

    // q in registers: for every head of a pass, the lane's CPL chunks (chunk pp + 8 j)
    float qr[Geo::NPASS][HG][CPL * EPL];
#pragma unroll
    for (int pa = 0; pa < Geo::NPASS; ++pa)
#pragma unroll
      for (int hh = 0; hh < HG; ++hh)
#pragma unroll
        for (int j = 0; j < CPL; ++j)
#pragma unroll
          for (int e = 0; e < EPL; ++e) qr[pa][hh][j * EPL + e] = qs[(pa * HG + hh) * D + (pp + LPR * j) * EPL + e];

    // per pass: the reference (lazy running max, log2 units) of the lane's head,
    // and its normaliser (writer lanes)
    float mh[Geo::NPASS], zl[Geo::NPASS];
    float2 o[G][EV / 2];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < EV / 2; ++e) o[g][e] = make_float2(0.f, 0.f);
#pragma unroll
    for (int pa = 0; pa < Geo::NPASS; ++pa) {
      mh[pa] = -INFINITY;
      zl[pa] = 0.f;
    }
    float *lgu = ws.lgw + u * (long)G * (cap + 1);
    const T *vn = v_new + u * (long)D;

    for (; gb < item_end; ++gb, ++i) {
      if (!ok) continue;
      const int r0 = static_cast<int>(gb % NB) * RB;
      const int rows = max(0, min(RB, n - r0));                // cached rows of the block
      const bool has_new = nc > n && n >= r0 && n < r0 + RB;  // the new token is block row `rows`
      const bool my_new = has_new && rows >= wr0 && rows < wr0 + RPW;  // ... and one of this warp's
      const int wrows = max(0, min(RPW, rows - wr0));          // this warp's cached rows
      const int wnv = wrows + (my_new ? 1 : 0);
      const int si = static_cast<int>(i % S);
      const uint32_t ph = static_cast<uint32_t>((i / S) & 1);

      // the new token's logits (every head): the lanes across d, then a warp sum
      float lnew[G];
      if (my_new) {
        const typename RP::Word word =
            __ldg(reinterpret_cast<const typename RP::Word *>(k_new + u * (long)D + lane * EV));
        float kv[EV];
        RP::unpack(word, kv);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float s = 0.f;
#pragma unroll
          for (int e = 0; e < EV; ++e) s = fmaf(kv[e], qs[g * D + lane * EV + e], s);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
          lnew[g] = c_log2 * s;
        }
      }

      if (!tc::mbar_wait(kfull + si, ph, kWaitBudget, abort_flag)) {
        fail(abort_flag, dev_status);
        ok = false;
        continue;
      }
      // K stage: LPR lanes per row, RPI rows per step; lane ends with one head's logit
      float l[Geo::NPASS][KIT];
      {
        const unsigned char *kst = sK + si * Geo::STAGE + (wr0 + rs) * Geo::ROWB + pp * 16;
#pragma unroll
        for (int it = 0; it < KIT; ++it) {
          float f[CPL][EPL];
#pragma unroll
          for (int j = 0; j < CPL; ++j)
            Vec16<T>::unpack(*reinterpret_cast<const uint4 *>(kst + RPI * it * Geo::ROWB + LPR * j * 16), f[j]);
#pragma unroll
          for (int pa = 0; pa < Geo::NPASS; ++pa) {
            float v[HG];
#pragma unroll
            for (int hh = 0; hh < HG; ++hh) {
              float2 part = make_float2(0.f, 0.f);
#pragma unroll
              for (int j = 0; j < CPL; ++j)
#pragma unroll
                for (int e = 0; e < EPL; e += 2)
                  part = __ffma2_rn(make_float2(f[j][e], f[j][e + 1]),
                                    make_float2(qr[pa][hh][j * EPL + e], qr[pa][hh][j * EPL + e + 1]), part);
              v[hh] = part.x + part.y;
            }
            l[pa][it] = c_log2 * row_butterfly<HG>(v, pp);
          }
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(kempty + si);
      if (my_new) {
        const int rn = rows - wr0;  // the new token's row among this warp's
#pragma unroll
        for (int it = 0; it < KIT; ++it)
          if (RPI * it + rs == rn)
#pragma unroll
            for (int pa = 0; pa < Geo::NPASS; ++pa)
#pragma unroll
              for (int hh = 0; hh < HG; ++hh)
                if (hh == hd) l[pa][it] = lnew[pa * HG + hh];
      }
      // logits to the workspace; per head, weights 2^(l - reference) with a lazy reference
#pragma unroll
      for (int pa = 0; pa < Geo::NPASS; ++pa) {
        float bm = -INFINITY;
#pragma unroll
        for (int it = 0; it < KIT; ++it) {
          const int rr = RPI * it + rs;  // row among this warp's
          if (rr < wnv) {
            bm = fmaxf(bm, l[pa][it]);
            if (writer) lgu[(long)(pa * HG + hd) * (cap + 1) + r0 + wr0 + rr] = l[pa][it];
          }
        }
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, off));
        // a new reference only when the block's max passes the old one by more than
        // kLazyLog2 (or on the first rows): weights stay below 2^kLazyLog2
        float s = 1.f;
        if (bm > mh[pa] + kLazyLog2) {
          s = tc::ex2(mh[pa] - bm);  // 0 while nothing has been seen
          zl[pa] *= s;
          mh[pa] = bm;
        }
#pragma unroll
        for (int hh = 0; hh < HG; ++hh) {
          const float sh = __shfl_sync(0xFFFFFFFFu, s, hh * DUP);  // lane hh * DUP holds head hh
          if (sh != 1.f) {
#pragma unroll
            for (int e = 0; e < EV / 2; ++e) o[pa * HG + hh][e] = __fmul2_rn(o[pa * HG + hh][e], make_float2(sh, sh));
          }
        }
#pragma unroll
        for (int it = 0; it < KIT; ++it) {
          const int rr = RPI * it + rs;
          const float p = rr < wnv ? tc::ex2(l[pa][it] - mh[pa]) : 0.f;
          if (writer) {
            zl[pa] += p;
            pww[rr * G + pa * HG + hd] = p;
          }
        }
      }
      __syncwarp();

      // V stage: one row at a time across the lanes
      if (!tc::mbar_wait(vfull + si, ph, kWaitBudget, abort_flag)) {
        fail(abort_flag, dev_status);
        ok = false;
        continue;
      }
      {
        const unsigned char *vst = sV + si * Geo::STAGE + wr0 * Geo::ROWB + lane * EV * (int)sizeof(T);
        auto accum = [&](const typename RP::Word &word, int r) {
          float vv[EV];
          RP::unpack(word, vv);
          float pg[G];
          if constexpr (G % 4 == 0) {
#pragma unroll
            for (int g4 = 0; g4 < G; g4 += 4) {
              const float4 p4 = *reinterpret_cast<const float4 *>(pww + r * G + g4);
              pg[g4] = p4.x;
              pg[g4 + 1] = p4.y;
              pg[g4 + 2] = p4.z;
              pg[g4 + 3] = p4.w;
            }
          } else {
#pragma unroll
            for (int g = 0; g < G; ++g) pg[g] = pww[r * G + g];
          }
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < EV / 2; ++e)
              o[g][e] = __ffma2_rn(make_float2(pg[g], pg[g]), make_float2(vv[2 * e], vv[2 * e + 1]), o[g][e]);
        };
        if (wrows == RPW) {
#pragma unroll
          for (int r8 = 0; r8 < RPW; r8 += 8) {
            typename RP::Word word[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              word[k] = *reinterpret_cast<const typename RP::Word *>(vst + (r8 + k) * Geo::ROWB);
#pragma unroll
            for (int k = 0; k < 8; ++k) accum(word[k], r8 + k);
          }
        } else {
          for (int r = 0; r < wrows; ++r) accum(*reinterpret_cast<const typename RP::Word *>(vst + r * Geo::ROWB), r);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(vempty + si);
        if (my_new) accum(__ldg(reinterpret_cast<const typename RP::Word *>(vn + lane * EV)), wrows);
      }
      __syncwarp();  // pww is rewritten by the next block
    }

    // ---- the unit's range in this CTA is done: combine the warps into one partial ----
    float *pbw = pb + w * PBW;
#pragma unroll
    for (int pa = 0; pa < Geo::NPASS; ++pa) {
      float z = writer ? zl[pa] : 0.f;
      // lanes with the same head: the same pp / DUP in every row group
#pragma unroll
      for (int off = LPR; off < 32; off <<= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, off);
#pragma unroll
      for (int off = 1; off < DUP; off <<= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, off);
      if (lane < LPR && writer) {
        pbw[G * D + G + pa * HG + hd] = z;
        pbw[G * D + pa * HG + hd] = mh[pa];
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < EV / 2; ++e) {
        pbw[g * D + lane * EV + 2 * e] = o[g][e].x;
        pbw[g * D + lane * EV + 2 * e + 1] = o[g][e].y;
      }
    tc::named_bar_sync(BAR_CONS, NCT);
    if (ct < G) {
      float M = -INFINITY;
      for (int v = 0; v < NCW; ++v) M = fmaxf(M, pb[v * PBW + G * D + ct]);
      float Z = 0.f;
      for (int v = 0; v < NCW; ++v) {
        const float mv = pb[v * PBW + G * D + ct];
        const float sv = mv == -INFINITY ? 0.f : tc::ex2(mv - M);
        sc[v * G + ct] = sv;
        Z += pb[v * PBW + G * D + G + ct] * sv;
      }
      fm[ct] = M;
      fz[ct] = Z;
    }
    tc::named_bar_sync(BAR_CONS, NCT);
    const Span sp = unit_span(u, NB, per);
    const long slot = u * PM + (static_cast<int>(blockIdx.x) - sp.first);
    float *pou = ws.po + slot * (long)G * D;
    for (int t = ct; t < G * D; t += NCT) {
      const int g = t / D;
      float s = 0.f;
      for (int v = 0; v < NCW; ++v) s += pb[v * PBW + t] * sc[v * G + g];
      pou[t] = s;
    }
    if (ct < G) ws.pmz[slot * G + ct] = make_float2(fm[ct], fz[ct]);
  }
}

// Two entry points with one body.  For G <= 4 a stream thread gets at most 144
// registers and a finalize thread at most 80, so that a finalize CTA of the
// other half of the rows fits on the SM beside a stream CTA: the stream CTA's
// nine warps put three on one SM sub-partition, and 3 x 144 + 80 registers a
// lane fill that sub-partition's 16K-register file exactly (at 168 the stream
// warps leave 256 registers, and the finalize CTAs had to wait for the stream
// CTAs to leave).  G = 8 keeps the full budget in both kernels.
#define KVC_STREAM_PARAMS                                                                          \
  const T *__restrict__ Kc, const T *__restrict__ Vc, const T *__restrict__ q,                     \
      const T *__restrict__ k_new, const T *__restrict__ v_new, const int32_t *__restrict__ len,   \
      int Hq, int Hkv, int cap, float c_log2, int alg1, long total, long per, Ws ws,               \
      int *__restrict__ dev_status
#define KVC_STREAM_ARGS Kc, Vc, q, k_new, v_new, len, Hq, Hkv, cap, c_log2, alg1, total, per, ws, dev_status
template <typename T, int D, int G>
__global__ __maxnreg__(144) void decode_stream_kernel(KVC_STREAM_PARAMS) {
  decode_stream_body<T, D, G>(KVC_STREAM_ARGS);
}
template <typename T, int D, int G>
__global__ __launch_bounds__(32 * (NCW + 1), 1) void decode_stream_kernel_wide(KVC_STREAM_PARAMS) {
  decode_stream_body<T, D, G>(KVC_STREAM_ARGS);
}
#undef KVC_STREAM_PARAMS
#undef KVC_STREAM_ARGS

template <typename T, int D, int G>
__device__ __forceinline__ void decode_finalize_body(
    const T *__restrict__ k_new, const T *__restrict__ v_new, T *__restrict__ Kc, T *__restrict__ Vc,
    int32_t *__restrict__ pos, float *__restrict__ acc, int32_t *__restrict__ len, int Hq, int Hkv,
    int cap, int recent, int sink, int new_pos, int alg1, long per, Ws ws, float *__restrict__ o_out,
    int32_t *__restrict__ evicted, int *__restrict__ dev_status) {
  constexpr int NWF = NTF / 32;
  constexpr int GD = G * D;
  __shared__ float gm[G], gz[G], gc[G];
  __shared__ Cand wc[NWF];
  __shared__ int sh_slot, sh_last;
  const int rank = static_cast<int>(blockIdx.x % CE);
  const long unit = blockIdx.x / CE;
  const long b = unit / Hkv;
  const int h = static_cast<int>(unit % Hkv);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int NB = blocks_per_unit(cap, DGeo<T, D, G>::RB);
  const int PM = partials_per_unit(cap);
  const Span sp = unit_span(unit, NB, per);
  const float2 *pmz = ws.pmz + unit * PM * G;
  const float *po = ws.po + unit * PM * (long)GD;
  const float *lgu = ws.lgw + unit * (long)G * (cap + 1);
  float *au = acc + unit * (long)cap;
  int32_t *pu = pos + unit * (long)cap;

  // Every load that does not depend on the unit's length is issued before it is
  // known, so that a CTA waits for about one memory round trip, not three: the
  // length, the partials (m, Z) and this thread's output shares, and this CTA's
  // slots.  Slots are shared out by capacity (cap + 1 attended rows at most);
  // rows past the length are loaded (in bounds) and ignored.
  const int n_raw = len[unit];
  constexpr int PR = 4;  // partials held in registers; a longer span reads the rest in a loop
  const int t_out = rank * (GD / CE) + static_cast<int>(threadIdx.x);  // this thread's output
  const bool has_out = threadIdx.x < GD / CE;
  const int g_out = t_out / D;
  float2 mzr[PR];
  float2 mzo[PR];
  float por[PR];
#pragma unroll
  for (int p = 0; p < PR; ++p) {
    const bool pin = p < sp.count;
    mzr[p] = (pin && threadIdx.x < G) ? pmz[p * G + threadIdx.x] : make_float2(-INFINITY, 0.f);
    mzo[p] = (pin && has_out) ? pmz[p * G + g_out] : make_float2(-INFINITY, 0.f);
    por[p] = (pin && has_out) ? po[(long)p * GD + t_out] : 0.f;
  }
  const int ncap = cap + 1;
  const int per_cta = (ncap + CE - 1) / CE;
  const int j0 = min(ncap, rank * per_cta), j1c = min(ncap, j0 + per_cta);
  float lv[RU][G], av[RU];
  int pv[RU];
  auto load_slots = [&](int jb) {
#pragma unroll
    for (int k = 0; k < RU; ++k) {
      const int j = jb + k * NTF;
      if (j < j1c) {
#pragma unroll
        for (int g = 0; g < G; ++g) lv[k][g] = lgu[(long)g * (cap + 1) + j];
        if (j < cap) {
          av[k] = au[j];
          pv[k] = pu[j];
        }
      }
    }
  };
  const int jstart = j0 + threadIdx.x;
  load_slots(jstart);

  const int n = n_raw;
  if (n < 0 || n > cap) {  // same n in all the unit's CTAs: every one leaves here
    if (rank == 0 && threadIdx.x == 0 && dev_status) atomicExch(dev_status, (int)KV_ERR_INVALID_ARG);
    return;
  }
  const int nc = n + (alg1 ? 0 : 1);
  const int j1 = min(nc, j1c);
  // the unit's max and normaliser per head over the partials (a partial of an
  // empty range has m = -inf and Z = 0 and adds nothing)
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    float M = -INFINITY, Z = 0.f;
    auto add = [&](float2 v) {
      if (v.x == -INFINITY) return;
      const float Mn = fmaxf(M, v.x);
      Z = Z * tc::ex2(M - Mn) + v.y * tc::ex2(v.x - Mn);
      M = Mn;
    };
#pragma unroll
    for (int p = 0; p < PR; ++p)
      if (p < sp.count) add(mzr[p]);
    for (int p = PR; p < sp.count; ++p) add(pmz[p * G + g]);
    gm[g] = M;
    gz[g] = Z;
    gc[g] = M + log2f(Z);  // 2^(l - M) / Z = 2^(l - gc)
  }
  __syncthreads();
  // this CTA's part of the output: o_g = sum_p o_p exp(m_p - M) / Z
  float *ou = o_out + (b * Hq + (long)h * G) * D;
  // (the thread's first output has its shares in registers; o_p = 0 where m_p = -inf)
  for (int t = t_out, it = 0; t < (rank + 1) * (GD / CE); t += NTF, ++it) {
    const int g = t / D;
    float s = 0.f;
    int p = 0;
    if (it == 0) {
#pragma unroll
      for (int q = 0; q < PR; ++q)
        if (q < sp.count) s += por[q] * (mzo[q].x == -INFINITY ? 0.f : tc::ex2(mzo[q].x - gm[g]));
      p = PR;
    }
    for (; p < sp.count; ++p) {
      const float mp = pmz[p * G + g].x;
      s += po[(long)p * GD + t] * (mp == -INFINITY ? 0.f : tc::ex2(mp - gm[g]));
    }
    ou[t] = nc > 0 ? s / gz[g] : 0.f;
  }
  // probabilities -> accumulators, eviction candidate
  const long lim = (long)new_pos - recent;
  float best_a = INFINITY;
  int best_p = 0x7FFFFFFF, best_j = -2;
  float acc_self = 0.f;
  for (int jb = jstart; jb < j1; jb += RU * NTF) {
    if (jb != jstart) load_slots(jb);
#pragma unroll
    for (int k = 0; k < RU; ++k) {
      const int j = jb + k * NTF;
      if (j >= j1) continue;
      float P = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g) P += tc::ex2(lv[k][g] - gc[g]);
      if (j < n) {
        const float a = av[k] + P;
        au[j] = a;
        if ((long)pv[k] <= lim && pv[k] >= sink && better(a, pv[k], best_a, best_p)) {
          best_a = a;
          best_p = pv[k];
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
    for (int v = 0; v < NWF; ++v) {
      if (wc[v].slot != -2 && (c.slot == -2 || better(wc[v].acc, wc[v].pos, c.acc, c.pos))) {
        c.acc = wc[v].acc;
        c.pos = wc[v].pos;
        c.slot = wc[v].slot;
      }
      c.accself += wc[v].accself;
    }
    // publish this CTA's candidate; the unit's last CTA to arrive decides
    ws.cnd[unit * CE + rank] = c;
    __threadfence();
    sh_last = atomicAdd(ws.cnt + unit, 1) == CE - 1;
  }
  __syncthreads();
  if (!sh_last) return;
  if (threadIdx.x == 0) {
    __threadfence();
    float ba = INFINITY, accnew = 0.f;
    int bp = 0x7FFFFFFF, bj = -2;
    for (int r = 0; r < CE; ++r) {
      const float4 raw = __ldcg(reinterpret_cast<const float4 *>(ws.cnd + unit * CE + r));
      const Cand cc{raw.x, __float_as_int(raw.y), __float_as_int(raw.z), raw.w};
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
    constexpr int VECS = D * (int)sizeof(T) / 16;
    uint4 *kd = reinterpret_cast<uint4 *>(Kc + (unit * (long)cap + slot) * D);
    uint4 *vd = reinterpret_cast<uint4 *>(Vc + (unit * (long)cap + slot) * D);
    const uint4 *ks = reinterpret_cast<const uint4 *>(k_new + unit * (long)D);
    const uint4 *vs = reinterpret_cast<const uint4 *>(v_new + unit * (long)D);
    for (int t = threadIdx.x; t < VECS; t += NTF) {
      kd[t] = __ldg(ks + t);
      vd[t] = __ldg(vs + t);
    }
  }
}

#define KVC_FIN_PARAMS                                                                             \
  const T *__restrict__ k_new, const T *__restrict__ v_new, T *__restrict__ Kc,                    \
      T *__restrict__ Vc, int32_t *__restrict__ pos, float *__restrict__ acc,                      \
      int32_t *__restrict__ len, int Hq, int Hkv, int cap, int recent, int sink, int new_pos,      \
      int alg1, long per, Ws ws, float *__restrict__ o_out, int32_t *__restrict__ evicted,         \
      int *__restrict__ dev_status
#define KVC_FIN_ARGS                                                                               \
  k_new, v_new, Kc, Vc, pos, acc, len, Hq, Hkv, cap, recent, sink, new_pos, alg1, per, ws, o_out,   \
      evicted, dev_status
template <typename T, int D, int G>
__global__ __maxnreg__(80) void decode_finalize_kernel(KVC_FIN_PARAMS) {
  decode_finalize_body<T, D, G>(KVC_FIN_ARGS);
}
template <typename T, int D, int G>
__global__ __launch_bounds__(NTF) void decode_finalize_kernel_wide(KVC_FIN_PARAMS) {
  decode_finalize_body<T, D, G>(KVC_FIN_ARGS);
}
#undef KVC_FIN_PARAMS
#undef KVC_FIN_ARGS

template <typename T, int D, int G>
int run_decode(const void *q, const void *k_new, const void *v_new, void *K_cache, void *V_cache,
               int32_t *pos, float *acc, int32_t *len, int B, int Hq, int Hkv, int cap,
               int recent, int sink, int new_pos, float scale, int flags, void *workspace, float *o,
               int32_t *evicted, int *dev_status, cudaStream_t st) {
  using Geo = DGeo<T, D, G>;
  const long units = (long)B * Hkv;
  const Ws ws = carve(workspace, units, G, cap, D);
  const int alg1 = (flags & KV_H2O_ALG1) ? 1 : 0;
  auto stream_kernel = [] {
    if constexpr (G <= 4) {
      return decode_stream_kernel<T, D, G>;
    } else {
      return decode_stream_kernel_wide<T, D, G>;
    }
  }();
  auto finalize_kernel = [] {
    if constexpr (G <= 4) {
      return decode_finalize_kernel<T, D, G>;
    } else {
      return decode_finalize_kernel_wide<T, D, G>;
    }
  }();
  if (ensure_smem((const void *)stream_kernel, Geo::SMEM))
    return cuda_failure(cudaErrorInvalidValue, "decode stream kernel: shared memory limit");
  const int NB = blocks_per_unit(cap, Geo::RB);
  const long total = units * NB;
  const long grid = std::max(1L, std::min((long)device_sm_count(), total / PER_MIN));
  const long per = (total + grid - 1) / grid;
  const long ctas = (total + per - 1) / per;
  stream_kernel<<<(unsigned)ctas, 32 * (NCW + 1), Geo::SMEM, st>>>(
      static_cast<const T *>(K_cache), static_cast<const T *>(V_cache), static_cast<const T *>(q),
      static_cast<const T *>(k_new), static_cast<const T *>(v_new), len, Hq, Hkv, cap,
      scale * 1.4426950408889634f /* log2 e */, alg1, total, per, ws, dev_status);
  {
    const int rc = launch_status(0);  // the stream kernel's launch
    if (rc != KV_OK) return rc;
  }
  finalize_kernel<<<(unsigned)(units * CE), NTF, 0, st>>>(
      static_cast<const T *>(k_new), static_cast<const T *>(v_new), static_cast<T *>(K_cache),
      static_cast<T *>(V_cache), pos, acc, len, Hq, Hkv, cap, recent, sink, new_pos, alg1, per, ws, o, evicted,
      dev_status);
  return launch_status(2);
}

template <typename T, int D>
int dispatch_g(int G, const void *q, const void *k_new, const void *v_new, void *K_cache,
               void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq, int Hkv,
               int cap, int recent, int sink, int new_pos, float scale, int flags, void *workspace,
               float *o, int32_t *evicted, int *dev_status, cudaStream_t st) {
#define KVC_DEC(GG)                                                                          \
  if (G == GG)                                                                               \
    return run_decode<T, D, GG>(q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq, Hkv, \
                                cap, recent, sink, new_pos, scale, flags, workspace, o, evicted,    \
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
  const int PM = partials_per_unit(cap);
  return align256((size_t)units * G * (cap + 1) * 4) + align256((size_t)units * PM * G * 8) +
         align256((size_t)units * PM * G * d * 4) + align256((size_t)units * CE * sizeof(Cand)) +
         (size_t)units * sizeof(int);
}

int launch_decode_step(const void *q, const void *k_new, const void *v_new, void *K_cache,
                       void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq,
                       int Hkv, int cap, int d, int recent, int sink, int32_t new_pos, float scale,
                       int flags, int dtype, void *workspace, float *o, int32_t *evicted,
                       int *dev_status, cudaStream_t st) {
  const int G = Hq / Hkv;
  if (dtype == KV_BF16) {
    if (d == 128)
      return dispatch_g<__nv_bfloat16, 128>(G, q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq,
                                            Hkv, cap, recent, sink, new_pos, scale, flags, workspace, o,
                                            evicted, dev_status, st);
    return dispatch_g<__nv_bfloat16, 64>(G, q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq,
                                         Hkv, cap, recent, sink, new_pos, scale, flags, workspace, o,
                                         evicted, dev_status, st);
  }
  if (d == 128)
    return dispatch_g<float, 128>(G, q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq, Hkv,
                                  cap, recent, sink, new_pos, scale, flags, workspace, o, evicted,
                                  dev_status, st);
  return dispatch_g<float, 64>(G, q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq, Hkv,
                               cap, recent, sink, new_pos, scale, flags, workspace, o, evicted,
                               dev_status, st);
}

}  // namespace kvc
