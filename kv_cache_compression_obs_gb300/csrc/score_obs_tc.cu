// score_obs_tc.cu -- observation-window scoring on the 5th-generation tensor cores.
//
// Same quantity as score_obs.cu (the accumulated attention of the H2O page,
// 观察二, over SnapKV's observation window, KV-cache blog §4.3), for bf16 inputs
// with G*W <= 256 query rows per unit (every GQA / MHA prefill workload).
// The logits are produced by tcgen05.mma (bf16 x bf16 -> fp32 in TMEM) from
// TMA-staged, 128-byte-swizzled shared-memory tiles:
//
//   pass 1 (statistics): D[rows x keys] = Q K^T with the query rows on the TMEM
//     lanes, so every epilogue thread owns one row and keeps its running max and
//     normaliser in registers (no cross-thread reduction);
//   combine: per row M = max and 1/Z over the key splits (score_obs.cu);
//   pass 2 (column mass): D[keys x rows] = K Q^T with the keys on the TMEM lanes,
//     so every epilogue thread owns one key and sums 2^(x - M_r) / Z_r over the
//     rows in registers.
//
// Both kernels are persistent (one CTA per SM, items assigned round-robin) and
// warp-specialised: warp 0 issues TMA loads into a 4-stage K ring (the unit's Q
// block stays resident per item), warp 1 issues the MMAs into two TMEM slots,
// warps 2..17 (four warpgroups, each taking a quarter of a tile's TMEM columns)
// drain TMEM.  Every mbarrier wait is bounded; a
// wait that gives up sets a CTA-wide abort flag and the device status
// KV_ERR_TIMEOUT, the roles leave their loops, outstanding copies and MMAs are
// waited for (again bounded) and the TMEM is freed before the CTA exits.
#include <cmath>

#include "kvc_internal.cuh"
#include "tc_common.cuh"

namespace kvc {
namespace {

constexpr int EPI_WARPS = 16;  // TMEM-draining warps (four warpgroups)
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int NT = 64 + EPI_THREADS;  // + producer warp + MMA warp
constexpr int KT = 128;        // keys per tile (the UMMA M of pass 2, N of pass 1)
constexpr int QROWS = 256;     // resident query rows per unit
constexpr int STAGES = 4;      // K ring depth
constexpr int TMEM_COLS = 512;
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (~2 s) before a wait gives up
constexpr long long kDrainBudget = 200000000LL;  // ~0.1 s for in-flight copies / MMAs at exit

template <int D>
struct Geo {
  static constexpr int NKB = D / 64;                  // 128-byte k-blocks per row
  static constexpr int KBYTES = KT * D * 2;           // one K tile
  static constexpr int QBYTES = QROWS * D * 2;        // resident Q block
  static constexpr int KSUB = KT * 128;               // bytes of one k-block of a K tile
  static constexpr int QSUB = QROWS * 128;            // bytes of one k-block of the Q block
  static constexpr int BAR_OFF = QBYTES + STAGES * KBYTES;   // 1024-aligned
  // barriers: full[S], empty[S], qfull, qempty, tfull[2], tempty[2], drain
  static constexpr int NBARS = 2 * STAGES + 7;
  static constexpr int MISC_OFF = BAR_OFF + 256;              // TMEM base, abort flag
  static constexpr int STAT_OFF = BAR_OFF + 512;              // row M, 1/Z, position (16-aligned)
  static constexpr int RED_OFF = STAT_OFF + QROWS * 12;       // warpgroup exchange (4 KB)
  // at least 116 KB so that a single CTA fits per SM: each CTA takes all 512 TMEM columns
  static constexpr int SMEM_NEED = 1024 /*alignment slack*/ + RED_OFF + 4096;
  static constexpr int SMEM = SMEM_NEED > 116 * 1024 ? SMEM_NEED : 116 * 1024;
  static_assert(NBARS * 8 <= 256, "barrier area");
};

struct Bars {
  uint64_t *full, *empty, *qfull, *qempty, *tfull, *tempty, *drain;
};

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
  return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ Bars carve_bars(unsigned char *base) {
  uint64_t *b = reinterpret_cast<uint64_t *>(base);
  return Bars{b, b + STAGES, b + 2 * STAGES, b + 2 * STAGES + 1, b + 2 * STAGES + 2,
              b + 2 * STAGES + 4, b + 2 * STAGES + 6};
}

__device__ __forceinline__ void init_bars(const Bars &B) {
  for (int i = 0; i < STAGES; ++i) {
    tc::mbar_init(B.full + i, 1);
    tc::mbar_init(B.empty + i, 1);
  }
  tc::mbar_init(B.qfull, 1);
  tc::mbar_init(B.qempty, 1);
  for (int i = 0; i < 2; ++i) {
    tc::mbar_init(B.tfull + i, 1);
    tc::mbar_init(B.tempty + i, EPI_WARPS);  // one arrival per epilogue warp
  }
  tc::mbar_init(B.drain, 1);
  tc::mbar_fence_init();
}

// Work decomposition shared by the three roles: item -> (unit, key range).
struct Item {
  long unit;
  int j_begin, j_end;  // keys [j_begin, j_end)
};
__device__ __forceinline__ Item item_of(int item, int per_unit, int span, int T) {
  Item it;
  it.unit = item / per_unit;
  const int c = item % per_unit;
  it.j_begin = c * span;
  it.j_end = min(T, it.j_begin + span);
  return it;
}

__device__ __forceinline__ void set_abort(volatile int *abort_flag, int *status) {
  *abort_flag = 1;
  if (status) atomicExch(status, (int)KV_ERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Producer (warp 0, one lane): Q block per item, K tiles through the ring.
// ---------------------------------------------------------------------------
template <int D>
__device__ void produce(const CUtensorMap *tmQ, const CUtensorMap *tmK, unsigned char *sQ,
                        unsigned char *sK, const Bars &B, int n_items, int per_unit, int span,
                        int Hq, int Hkv, int T, int W, volatile int *abort_flag, int *status) {
  using G = Geo<D>;
  tc::tma_prefetch_desc(tmQ);
  tc::tma_prefetch_desc(tmK);
  const int Gq = Hq / Hkv;
  uint32_t g = 0;
  int it = 0;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
    const Item w = item_of(item, per_unit, span, T);
    const long b = w.unit / Hkv;
    const int h = static_cast<int>(w.unit % Hkv);
    const int qrow0 = static_cast<int>((b * Hq + (long)h * Gq) * W);
    if (!tc::mbar_wait(B.qempty, (it & 1) ^ 1, kWaitBudget, abort_flag)) {
      set_abort(abort_flag, status);
      break;
    }
    tc::mbar_arrive_expect_tx(B.qfull, G::QBYTES);
    for (int kb = 0; kb < G::NKB; ++kb)
      for (int half = 0; half < 2; ++half)
        tc::tma_load_2d(sQ + kb * G::QSUB + half * 128 * 128, tmQ, kb * 64, qrow0 + half * 128, B.qfull);
    bool ok = true;
    for (int j0 = w.j_begin; j0 < w.j_end; j0 += KT, ++g) {
      const int st = g % STAGES;
      const uint32_t use = g / STAGES;
      if (!tc::mbar_wait(B.empty + st, (use & 1) ^ 1, kWaitBudget, abort_flag)) {
        set_abort(abort_flag, status);
        ok = false;
        break;
      }
      tc::mbar_arrive_expect_tx(B.full + st, G::KBYTES);
      const int krow = static_cast<int>(w.unit * (long)T + j0);
      for (int kb = 0; kb < G::NKB; ++kb)
        tc::tma_load_2d(sK + st * G::KBYTES + kb * G::KSUB, tmK, kb * 64, krow, B.full + st);
    }
    if (!ok) break;
  }
  // copies still in flight land before the CTA may exit: wait for the last
  // uses of every stage (bounded; completed phases return at once)
  for (int k = 1; k <= STAGES && (int)g - k >= 0; ++k) {
    const uint32_t gg = g - k;
    tc::mbar_wait(B.full + gg % STAGES, (gg / STAGES) & 1, kDrainBudget, nullptr);
  }
}

// ---------------------------------------------------------------------------
// MMA issuer (warp 1, one lane).  PASS 1: D[row, key] for the one or two
// 128-row M-tiles of Q.  PASS 2: D[key, row], N = n_cols query rows.
// ---------------------------------------------------------------------------
template <int D, int PASS>
__device__ void issue(uint32_t tmem, unsigned char *sQ, unsigned char *sK, const Bars &B,
                      int n_items, int per_unit, int span, int T, int n_mt, int n_cols,
                      volatile int *abort_flag, int *status) {
  using G = Geo<D>;
  // Operand descriptors: built once and stepped by constant offsets (the start
  // address field holds addr >> 4; shared memory stays below 2^18 bytes, so a
  // step never carries out of it).  The issuing thread shares its SMSP with busy
  // epilogue warps, so every instruction saved here keeps the tensor pipe fed.
  const uint64_t qd0 = tc::sdesc_sw128(tc::smem_u32(sQ));
  const uint64_t kd_base = tc::sdesc_sw128(tc::smem_u32(sK));
  const uint32_t idesc = (PASS == 1) ? tc::idesc_bf16(128, KT) : tc::idesc_bf16(128, n_cols);
  const bool two_mt = n_mt > 1;
  uint32_t g = 0;
  int it = 0;
  bool ok = true;
  for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
    const Item w = item_of(item, per_unit, span, T);
    if (!tc::mbar_wait(B.qfull, it & 1, kWaitBudget, abort_flag)) {
      set_abort(abort_flag, status);
      break;
    }
    tc::fence_after_sync();
    for (int j0 = w.j_begin; j0 < w.j_end; j0 += KT, ++g) {
      const int st = g % STAGES;
      const uint32_t use = g / STAGES;
      const int slot = g & 1;
      const uint32_t tuse = g >> 1;
      if (!tc::mbar_wait(B.full + st, use & 1, kWaitBudget, abort_flag) ||
          !tc::mbar_wait(B.tempty + slot, (tuse & 1) ^ 1, kWaitBudget, abort_flag)) {
        set_abort(abort_flag, status);
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint64_t kd0 = kd_base + (uint64_t)((st * G::KBYTES) >> 4);
      const uint32_t d0 = tmem + slot * 256;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t kd = kd0 + (uint64_t)(((kk / 4) * G::KSUB + (kk % 4) * 32) >> 4);
        const uint64_t qd = qd0 + (uint64_t)(((kk / 4) * G::QSUB + (kk % 4) * 32) >> 4);
        if (PASS == 1) {
          tc::umma_bf16(d0, qd, kd, idesc, kk > 0);
          if (two_mt) tc::umma_bf16(d0 + 128, qd + (uint64_t)((128 * 128) >> 4), kd, idesc, kk > 0);
        } else {
          tc::umma_bf16(d0, kd, qd, idesc, kk > 0);
        }
      }
      tc::umma_commit(B.empty + st);
      tc::umma_commit(B.tfull + slot);
    }
    if (ok) tc::umma_commit(B.qempty);
  }
  // every MMA issued above completes before TMEM can be released
  tc::umma_commit(B.drain);
  tc::mbar_wait(B.drain, 0, kDrainBudget, nullptr);
}

// Sums above this force the exact-max path of the statistics epilogue: every
// term is then at most 2^64, so the running normaliser cannot overflow.
constexpr float kLazyLimit = 1.8446744e19f;

// sum_c 2^(x_c * c_log2 - m) over 64 logits, two at a time with packed fp32 math.
__device__ __forceinline__ float chunk_sum(const uint32_t (&r)[64], float c_log2, float m) {
  const float2 c2 = make_float2(c_log2, c_log2);
  const float2 nm2 = make_float2(-m, -m);
  float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 64; c += 4) {
    const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), c2, nm2);
    const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(r[c + 2]), __uint_as_float(r[c + 3])), c2, nm2);
    a0 = __fadd2_rn(a0, make_float2(tc::ex2(x0.x), tc::ex2(x0.y)));
    a1 = __fadd2_rn(a1, make_float2(tc::ex2(x1.x), tc::ex2(x1.y)));
  }
  const float2 a = __fadd2_rn(a0, a1);
  return a.x + a.y;
}

// ---------------------------------------------------------------------------
// Pass 1: per-row running max and normaliser over a key split.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(NT, 1)
    score_stats_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          int Hq, int Hkv, int T, int W, int gw, int per_unit, int span, int n_items,
                          float c_log2, float2 *__restrict__ part, int *__restrict__ status) {
  using G = Geo<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  unsigned char *sQ = sm;
  unsigned char *sK = sm + G::QBYTES;
  const Bars B = carve_bars(sm + G::BAR_OFF);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + G::MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_mt = gw > 128 ? 2 : 1;

  if (threadIdx.x == 0) {
    init_bars(B);
    *abort_flag = 0;
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0)
      produce<D>(&tmQ, &tmK, sQ, sK, B, n_items, per_unit, span, Hq, Hkv, T, W, abort_flag, status);
  } else if (warp == 1) {
    if (lane == 0)
      issue<D, 1>(tmem, sQ, sK, B, n_items, per_unit, span, T, n_mt, 0, abort_flag, status);
  } else {
    const int ew = warp - 2;                // 0 .. EPI_WARPS-1
    const int wg = ew >> 2;                 // warpgroup 0..3
    const int mt = wg >> 1;                 // M-tile (rows 0..127 or 128..255)
    const int chalf = wg & 1;               // which 64 keys of each 128-key tile
    const int quarter = warp & 3;           // TMEM lane quarter this warp may access
    const int rit = quarter * 32 + lane;    // row within the M-tile
    const int row = mt * 128 + rit;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    float2 *xch = reinterpret_cast<float2 *>(sm + G::RED_OFF);  // [2 items][2 M-tiles][128]
    uint32_t g = 0;
    bool ok = true;
    int it = 0;
    // A warp that gives up keeps walking the same items and tiles (without
    // touching TMEM) so that every named barrier is reached by all epilogue threads.
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
      const Item w = item_of(item, per_unit, span, T);
      const int p_row = T - W + (row % W);
      const int jlim = min(w.j_end, p_row + 1);  // keys this row may see in the split
      float m = -INFINITY, z = 0.f;
      for (int j0 = w.j_begin; j0 < w.j_end; j0 += KT, ++g) {
        const int slot = g & 1;
        const uint32_t tuse = g >> 1;
        if (ok && !tc::mbar_wait(B.tfull + slot, tuse & 1, kWaitBudget, abort_flag)) {
          set_abort(abort_flag, status);
          ok = false;
        }
        if (!ok) continue;
        tc::fence_after_sync();
        if (mt < n_mt) {
          uint32_t r[64];
          const uint32_t col = tmem + lane_addr + slot * 256 + mt * 128 + chalf * 64;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            tc::tmem_ld16(col + q * 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16 * q]));
          tc::tmem_ld_wait();
          const int jb = j0 + chalf * 64;
          if (jb + 64 <= jlim) {
            // every key visible: sum against the running reference m; only a sum
            // large enough to risk overflow (or the first chunk, m = -inf) takes
            // the exact-max path
            float sum = chunk_sum(r, c_log2, m);
            if (!(sum <= kLazyLimit)) {
              float cm = -INFINITY;
#pragma unroll
              for (int c = 0; c < 64; ++c) cm = fmaxf(cm, __uint_as_float(r[c]));
              const float mnew = fmaxf(m, cm * c_log2);
              sum = chunk_sum(r, c_log2, mnew);
              z = z * tc::ex2(m - mnew);
              m = mnew;
            }
            z += sum;
          } else if (jb < jlim) {
            float cm = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (jb + c < jlim) cm = fmaxf(cm, __uint_as_float(r[c]));
            const float mnew = fmaxf(m, cm * c_log2);
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              const float e = tc::ex2(fmaf(__uint_as_float(r[c]), c_log2, -mnew));
              acc += (jb + c < jlim) ? e : 0.f;
            }
            z = z * tc::ex2(m - mnew) + acc;
            m = mnew;
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(B.tempty + slot);
      }
      // the two 64-key halves of each row meet here (buffer alternates per item)
      float2 *xb = xch + (it & 1) * 256;
      if (chalf == 1) xb[mt * 128 + rit] = make_float2(m, z);
      tc::named_bar_sync(1, EPI_THREADS);
      if (ok && chalf == 0 && mt < n_mt && row < gw) {
        const float2 o = xb[mt * 128 + rit];
        const float M = fmaxf(m, o.x);
        float Z = 0.f;
        if (m != -INFINITY) Z += z * tc::ex2(m - M);
        if (o.x != -INFINITY) Z += o.y * tc::ex2(o.x - M);
        const int split = item % per_unit;
        part[(w.unit * per_unit + split) * gw + row] = make_float2(M, Z);
      }
    }
  }
  __syncwarp();  // lanes that skipped a single-lane role rejoin their warp
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// acc2 += 2^(x_r c_log2 + m_r) over the 16 rows r of one TMEM chunk (m_r =
// -(M_r + log2 Z_r)); MASKED: only the rows whose position is at least the key's j.
template <bool MASKED>
__device__ __forceinline__ float2 colsum_chunk(const uint32_t (&r)[16], const float4 *m4, const int4 *p4, int j,
                                               float2 c2, float2 acc2) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float4 mm = m4[u];
    const float2 xa = __ffma2_rn(make_float2(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1])), c2,
                                 make_float2(mm.x, mm.y));
    const float2 xb = __ffma2_rn(make_float2(__uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3])), c2,
                                 make_float2(mm.z, mm.w));
    float2 ea = make_float2(tc::ex2(xa.x), tc::ex2(xa.y));
    float2 eb = make_float2(tc::ex2(xb.x), tc::ex2(xb.y));
    if constexpr (MASKED) {
      const int4 pp = p4[u];
      ea = make_float2(j <= pp.x ? ea.x : 0.f, j <= pp.y ? ea.y : 0.f);
      eb = make_float2(j <= pp.z ? eb.x : 0.f, j <= pp.w ? eb.y : 0.f);
    }
    acc2 = __fadd2_rn(acc2, __fadd2_rn(ea, eb));
  }
  return acc2;
}

// ---------------------------------------------------------------------------
// Pass 2: column mass s_j = sum_r 2^(x_rj - M_r - log2 Z_r) over a key chunk.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(NT, 1)
    score_colsum_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           int Hq, int Hkv, int T, int W, int gw, int n_cols, int per_unit, int span,
                           int n_items, float c_log2, const float2 *__restrict__ fin,
                           float *__restrict__ s_out, int *__restrict__ status) {
  using G = Geo<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  unsigned char *sQ = sm;
  unsigned char *sK = sm + G::QBYTES;
  const Bars B = carve_bars(sm + G::BAR_OFF);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + G::MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  float *sM = reinterpret_cast<float *>(sm + G::STAT_OFF);
  float *sZ = sM + QROWS;
  int *sPos = reinterpret_cast<int *>(sZ + QROWS);
  float *sRed = reinterpret_cast<float *>(sm + G::RED_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    init_bars(B);
    *abort_flag = 0;
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0)
      produce<D>(&tmQ, &tmK, sQ, sK, B, n_items, per_unit, span, Hq, Hkv, T, W, abort_flag, status);
  } else if (warp == 1) {
    if (lane == 0)
      issue<D, 2>(tmem, sQ, sK, B, n_items, per_unit, span, T, 0, n_cols, abort_flag, status);
  } else {
    const int et = threadIdx.x - 64;        // 0 .. EPI_THREADS-1
    const int ew = warp - 2;
    const int wg = ew >> 2;                 // this warpgroup takes column chunks wg, wg+4, ...
    const int quarter = warp & 3;
    const int key_in_tile = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const int n_chunks = n_cols / 16;
    const int first_masked = T - W;         // keys below this are seen by every row
    uint32_t g = 0;
    bool ok = true;
    // A warp that gives up keeps walking the same items and tiles (without
    // touching TMEM) so that every named barrier below is reached by all 256
    // epilogue threads.
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const Item w = item_of(item, per_unit, span, T);
      tc::named_bar_sync(1, EPI_THREADS);   // the previous item's readers are done
      for (int r = et; r < QROWS; r += EPI_THREADS) {
        if (r < gw) {
          const float2 f = fin[w.unit * gw + r];  // (M, 1/Z)
          // 2^(x c - M) / Z = 2^(x c - (M + log2 Z)); stored negated, so the
          // exponent is one fma: x * c_log2 + sM
          sM[r] = log2f(f.y) - f.x;
          sPos[r] = T - W + (r % W);
        } else {
          sM[r] = -INFINITY;  // padding rows contribute 2^-inf = 0
          sPos[r] = -1;
        }
      }
      tc::named_bar_sync(1, EPI_THREADS);
      for (int j0 = w.j_begin; j0 < w.j_end; j0 += KT, ++g) {
        const int slot = g & 1;
        const uint32_t tuse = g >> 1;
        if (ok && !tc::mbar_wait(B.tfull + slot, tuse & 1, kWaitBudget, abort_flag)) {
          set_abort(abort_flag, status);
          ok = false;
        }
        const int j = j0 + key_in_tile;
        float acc = 0.f;
        if (ok) {
          tc::fence_after_sync();
          const bool masked = j0 + KT > first_masked;
          float2 acc2 = make_float2(0.f, 0.f);
          const float2 c2 = make_float2(c_log2, c_log2);
          {
            // this warpgroup's (at most four) 16-column chunks in flight before one wait
            uint32_t r[4][16];
            const int nq = max(0, min(4, (n_chunks - wg + 3) / 4));
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (q < nq) tc::tmem_ld16(tmem + lane_addr + slot * 256 + (wg + 4 * q) * 16, r[q]);
            if (nq > 0) tc::tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (q >= nq) break;
              const int ch = wg + 4 * q;
              const float4 *m4 = reinterpret_cast<const float4 *>(sM + ch * 16);
              const int4 *p4 = reinterpret_cast<const int4 *>(sPos + ch * 16);
              acc2 = masked ? colsum_chunk<true>(r[q], m4, p4, j, c2, acc2)
                            : colsum_chunk<false>(r[q], m4, p4, j, c2, acc2);
            }
          }
          acc = acc2.x + acc2.y;
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(B.tempty + slot);
        }
        // add the four warpgroups' shares (fixed order) and store the key's mass;
        // the exchange buffer alternates between tiles, so one barrier per tile suffices
        float *red = sRed + (g & 1) * 4 * KT;
        if (wg > 0) red[wg * KT + key_in_tile] = acc;
        tc::named_bar_sync(1, EPI_THREADS);
        if (ok && wg == 0 && j < w.j_end)
          s_out[w.unit * (long)T + j] =
              acc + (red[KT + key_in_tile] + red[2 * KT + key_in_tile] + red[3 * KT + key_in_tile]);
      }
    }
  }
  __syncwarp();  // lanes that skipped a single-lane role rejoin their warp
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// rows x d bf16 matrix, boxes of 64 elements x 128 rows, 128-byte swizzle.
bool encode_rows(CUtensorMap *map, const void *base, long rows, int d) {
  return tc::encode_rows_sw128(map, base, rows, d, 2, 128);
}

template <int D>
int run_tc(const void *Q, const void *K, int B, int Hq, int Hkv, int T, int W, float scale,
           float *s, void *ws, const ScorePlan &plan, int *status, cudaStream_t st) {
  using G = Geo<D>;
  const long units = (long)B * Hkv;
  float2 *part = static_cast<float2 *>(ws);
  float2 *fin = part + units * plan.tc_splits * plan.gw;
  CUtensorMap tmQ, tmK;
  if (!encode_rows(&tmQ, Q, (long)B * Hq * W, D) || !encode_rows(&tmK, K, units * T, D))
    return KV_ERR_CUDA;
  if (ensure_smem((const void *)score_stats_tc_kernel<D>, G::SMEM) ||
      ensure_smem((const void *)score_colsum_tc_kernel<D>, G::SMEM))
    return KV_ERR_CUDA;
  const float c_log2 = scale * 1.4426950408889634f;
  const int sms = device_sm_count();
  const int n1 = (int)(units * plan.tc_splits);
  score_stats_tc_kernel<D><<<min(n1, sms), NT, G::SMEM, st>>>(
      tmQ, tmK, Hq, Hkv, T, W, plan.gw, plan.tc_splits, plan.tc_split_len, n1, c_log2, part, status);
  int rc = launch_score_combine(part, plan.tc_splits, plan.gw, units * plan.gw, fin, st);
  if (rc != KV_OK) return rc;
  const int n2 = (int)(units * plan.tc_splits);
  const int n_cols = ((plan.gw + 15) / 16) * 16;
  score_colsum_tc_kernel<D><<<min(n2, sms), NT, G::SMEM, st>>>(
      tmQ, tmK, Hq, Hkv, T, W, plan.gw, n_cols, plan.tc_splits, plan.tc_split_len, n2, c_log2, fin,
      s, status);
  return launch_status(2);
}

}  // namespace

bool score_tc_eligible(int dtype, int d, int Hq, int Hkv, int W) {
  const long gw = (long)(Hq / Hkv) * W;
  return dtype == KV_BF16 && (d == 64 || d == 128) && gw <= QROWS;
}

int launch_score_obs_tc(const void *Q, const void *K, int B, int Hq, int Hkv, int T, int d, int W,
                        float scale, float *s, void *ws, const ScorePlan &plan, int *status,
                        cudaStream_t st) {
  if (d == 128) return run_tc<128>(Q, K, B, Hq, Hkv, T, W, scale, s, ws, plan, status, st);
  return run_tc<64>(Q, K, B, Hq, Hkv, T, W, scale, s, ws, plan, status, st);
}

}  // namespace kvc
