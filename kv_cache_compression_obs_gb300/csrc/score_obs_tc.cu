// score_obs_tc.cu -- observation-window scoring on the 5th-generation tensor cores.
//
// Same quantity as score_obs.cu (the accumulated attention of the H2O page,
// 观察二, over SnapKV's observation window, KV-cache blog §4.3), for bf16 inputs.
// The logits are produced by tcgen05.mma (bf16 x bf16 -> fp32 in TMEM) from
// TMA-staged, 128-byte-swizzled shared-memory tiles.  A unit's G*W query rows
// are taken in row blocks of up to 256; each row block sees the keys up to its
// last row's position (causal), so the full-prompt scoring of the H2O page
// (every prompt query observed, W = T, 32 row blocks at T = 8192) is the same
// computation with more blocks.
//
// The exact column mass needs every row's softmax normaliser, so each logit is
// formed twice, by two persistent kernels over items (row block, key split):
//   statistics: D[rows x keys] = Q K^T with the query rows on the TMEM lanes;
//     every epilogue thread owns one row and keeps its running max and
//     normaliser in registers; the split's (max, sum) per row goes to the workspace;
//   merge: per row the exponent offset -(M + log2 Z) over the block's splits;
//   column mass: D[keys x rows] = K Q^T with the keys on the TMEM lanes; every
//     epilogue thread owns one key and sums 2^(x c - M_r - log2 Z_r) over the
//     block's rows.  With one row block per unit the kernel writes the scores;
//     with several it writes per-block column sums that a last kernel adds up in
//     block order (no float atomics: repeated runs give identical bits).
//
// Each kernel: one CTA per SM, items assigned round-robin; warp 0 issues TMA
// loads (a K tile ring of 4 stages; the row block's Q block, reloaded only when
// the block changes, after the first K tiles of the item are on their way),
// warp 1 issues the MMAs into two TMEM slots, warps 2..17 (four warpgroups,
// each taking a quarter of a tile's TMEM columns) drain TMEM.  Every mbarrier
// wait is bounded; a wait that gives up sets a CTA-wide abort flag and
// KV_ERR_TIMEOUT in the device status, the roles leave their loops,
// outstanding copies and MMAs are waited for (again bounded) and the TMEM is
// freed before the CTA exits.
#include <cmath>

#include "kvc_internal.cuh"
#include "tc_common.cuh"

namespace kvc {
namespace {

constexpr int EPI_WARPS = 16;  // TMEM-draining warps (four warpgroups)
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int NT = 64 + EPI_THREADS;  // + producer warp + MMA warp
constexpr int KT = 128;        // keys per tile (the UMMA M of the column pass, N of the statistics pass)
constexpr int QROWS = 256;     // query rows per row block
constexpr int STAGES = 4;      // K ring depth
constexpr int IRING = 4;       // claimed items the producer may run ahead of the consumers
constexpr int TMEM_COLS = 512;
constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (~2 s) before a wait gives up
constexpr long long kDrainBudget = 200000000LL;  // ~0.1 s for in-flight copies / MMAs at exit

template <int D>
struct Geo {
  static constexpr int NKB = D / 64;                  // 128-byte k-blocks per row
  static constexpr int KBYTES = KT * D * 2;           // one K tile
  static constexpr int QBYTES = QROWS * D * 2;        // one Q block
  static constexpr int KSUB = KT * 128;               // bytes of one k-block of a K tile
  static constexpr int QSUB = QROWS * 128;            // bytes of one k-block of the Q block
  static constexpr int BAR_OFF = QBYTES + STAGES * KBYTES;   // 1024-aligned
  // barriers: full[S], empty[S], qfull, qempty, tfull[2], tempty[2], drain, ifull[I], iempty[I]
  static constexpr int NBARS = 2 * STAGES + 7 + 2 * IRING;
  static constexpr int MISC_OFF = BAR_OFF + 256;              // TMEM base, abort flag, item ids
  static constexpr int STAT_OFF = BAR_OFF + 512;              // row offsets and positions (16-aligned)
  static constexpr int RED_OFF = STAT_OFF + QROWS * 8;        // warpgroup exchange (4 KB)
  static constexpr int SMEM_NEED = 1024 /*alignment slack*/ + RED_OFF + 4096;
  // at least 116 KB so that a single CTA fits per SM: each CTA takes all 512 TMEM columns
  static constexpr int SMEM = SMEM_NEED > 116 * 1024 ? SMEM_NEED : 116 * 1024;
  static_assert(NBARS * 8 <= 256, "barrier area");
};

struct Bars {
  uint64_t *full, *empty, *qfull, *qempty, *tfull, *tempty, *drain, *ifull, *iempty;
};

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
  return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ Bars carve_bars(unsigned char *base) {
  uint64_t *b = reinterpret_cast<uint64_t *>(base);
  return Bars{b, b + STAGES, b + 2 * STAGES, b + 2 * STAGES + 1, b + 2 * STAGES + 2,
              b + 2 * STAGES + 4, b + 2 * STAGES + 6, b + 2 * STAGES + 7, b + 2 * STAGES + 7 + IRING};
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
  for (int i = 0; i < IRING; ++i) {
    tc::mbar_init(B.ifull + i, 1);
    tc::mbar_init(B.iempty + i, 2);  // the MMA thread and the epilogue leader
  }
  tc::mbar_fence_init();
}

// Everything the kernels need to know about the call (passed by value).
struct Sched {
  int T, W, G, Hq, Hkv, gw;  // gw = G*W query rows per unit
  int nrb;                   // row blocks per unit
  int ns;                    // key splits per row block (over the whole prompt)
  int split_len;             // keys per split (a multiple of KT)
  int n_cols;                // UMMA N of the column pass
  int n_items;               // units * nrb * ns (splits past a block's last key are empty)
  int n_groups;              // units * nrb
  float c_log2;              // scale * log2(e)
  unsigned *next;            // this pass's claim counter (zeroed before the statistics pass)
  float2 *part;              // [groups][ns][QROWS] per-split (max, sum)
  const float *fin;          // [groups][QROWS] exponent offsets -(M + log2 Z)
  float *pcol;               // [units][nrb][T] per-block column sums (nrb > 1)
  float *s_out;              // [units][T]
  int *status;
};

// Row block g (unit-major): unit, block index, rows and the keys it sees.
struct Grp {
  int u;
  int rb, r0, nrows;
  int kend;    // keys [0, kend) are seen by some row of the block
  int kfull;   // keys below kfull are seen by every row of the block
  int nsplit;  // non-empty key splits
};
__host__ __device__ __forceinline__ Grp group_of(int g, int T, int W, int gw, int nrb,
                                                 int split_len) {
  Grp x;
  x.u = g / nrb;
  x.rb = g % nrb;
  x.r0 = x.rb * QROWS;
  x.nrows = gw - x.r0 < QROWS ? gw - x.r0 : QROWS;
  const int w0 = x.r0 % W;
  int wmin, wmax;
  if (w0 + x.nrows - 1 >= W) {  // the block passes the end of a query head's window
    wmin = 0;
    wmax = W - 1;
  } else {
    wmin = w0;
    wmax = w0 + x.nrows - 1;
  }
  x.kend = T - W + wmax + 1;
  x.kfull = T - W + wmin;
  x.nsplit = (x.kend + split_len - 1) / split_len;
  return x;
}

struct Item {
  int g;
  int ks, j0, j1;  // split index and its keys [j0, j1)
};
// Item index -> (row block, split): split-major, and within a split the row
// blocks that see the most keys first (all units' last blocks, then the
// blocks before them), so that claims take the largest items first and
// consecutive claims go to different units.  Returns false for a split past
// the block's last key.
__device__ __forceinline__ bool item_of(const Sched &S, int i, Item &it, Grp &grp) {
  it.ks = i / S.n_groups;
  const int r = i % S.n_groups;
  const int units = S.n_groups / S.nrb;
  it.g = (r % units) * S.nrb + (S.nrb - 1 - r / units);
  grp = group_of(it.g, S.T, S.W, S.gw, S.nrb, S.split_len);
  it.j0 = it.ks * S.split_len;
  it.j1 = min(it.j0 + S.split_len, grp.kend);
  return it.j0 < it.j1;
}

__device__ __forceinline__ void set_abort(volatile int *abort_flag, int *status) {
  *abort_flag = 1;
  if (status) atomicExch(status, (int)KV_ERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Producer (warp 0, one lane): the item's K tiles through the ring, and the row
// block's Q block when it changes (after the first K tiles: its buffer frees
// only when the previous item's MMAs have finished).
// ---------------------------------------------------------------------------
// Next non-empty item from the pass's claim counter, or -1 when none is left
// (or the CTA is aborting).
__device__ __forceinline__ int claim(const Sched &S, volatile int *abort_flag) {
  for (;;) {
    if (*abort_flag) return -1;
    const unsigned c = atomicAdd(S.next, 1u);
    if (c >= (unsigned)S.n_items) return -1;
    Item w;
    Grp grp;
    if (item_of(S, (int)c, w, grp)) return (int)c;
  }
}

template <int D>
__device__ void produce(const CUtensorMap *tmQ, const CUtensorMap *tmK, unsigned char *sQ,
                        unsigned char *sK, const Bars &B, int *ids, const Sched &S,
                        volatile int *abort_flag) {
  using Gm = Geo<D>;
  tc::tma_prefetch_desc(tmQ);
  tc::tma_prefetch_desc(tmK);
  uint32_t kt = 0, qv = 0;
  int prev_g = -1;
  bool ok = true;
  int next = claim(S, abort_flag);
  for (uint32_t it = 0;; ++it) {
    const int i = ok ? next : -1;
    const int slot = it % IRING;
    if (!tc::mbar_wait(B.iempty + slot, ((it / IRING) & 1) ^ 1, kWaitBudget, abort_flag)) {
      set_abort(abort_flag, S.status);
      ok = false;  // the consumers leave on the abort flag
    }
    ids[slot] = ok ? i : -1;
    tc::mbar_arrive(B.ifull + slot);
    if (i < 0 || !ok) break;
    next = claim(S, abort_flag);  // its latency overlaps this item's loads
    Item w;
    Grp grp;
    item_of(S, i, w, grp);
    const int ntiles = (w.j1 - w.j0 + KT - 1) / KT;
    const int krow0 = static_cast<int>((long long)grp.u * S.T + w.j0);
    auto load_k = [&](int t) {
      const int st = kt % STAGES;
      const uint32_t use = kt / STAGES;
      if (!tc::mbar_wait(B.empty + st, (use & 1) ^ 1, kWaitBudget, abort_flag)) {
        set_abort(abort_flag, S.status);
        ok = false;
        return;
      }
      tc::mbar_arrive_expect_tx(B.full + st, Gm::KBYTES);
      for (int kb = 0; kb < Gm::NKB; ++kb)
        tc::tma_load_2d(sK + st * Gm::KBYTES + kb * Gm::KSUB, tmK, kb * 64, krow0 + t * KT, B.full + st);
      ++kt;
    };
    int t = 0;
    if (w.g != prev_g) {
      prev_g = w.g;
      for (; t < ntiles && t < STAGES && ok; ++t) load_k(t);
      if (ok && !tc::mbar_wait(B.qempty, (qv & 1) ^ 1, kWaitBudget, abort_flag)) {
        set_abort(abort_flag, S.status);
        ok = false;
      }
      if (ok) {
        const long long b = grp.u / S.Hkv;
        const int h = grp.u % S.Hkv;
        const int qrow0 = static_cast<int>((b * S.Hq + (long long)h * S.G) * S.W + grp.r0);
        tc::mbar_arrive_expect_tx(B.qfull, Gm::QBYTES);
        for (int kb = 0; kb < Gm::NKB; ++kb)
          for (int half = 0; half < 2; ++half)
            tc::tma_load_2d(sQ + kb * Gm::QSUB + half * 128 * 128, tmQ, kb * 64, qrow0 + half * 128,
                            B.qfull);
        ++qv;
      }
    }
    for (; t < ntiles && ok; ++t) load_k(t);
  }
  // copies still in flight land before the CTA may exit: wait for the last uses
  // of every stage and the last Q block (bounded; completed phases return at once)
  for (int k = 1; k <= STAGES && (int)kt - k >= 0; ++k) {
    const uint32_t gg = kt - k;
    tc::mbar_wait(B.full + gg % STAGES, (gg / STAGES) & 1, kDrainBudget, nullptr);
  }
  if (qv > 0) tc::mbar_wait(B.qfull, (qv - 1) & 1, kDrainBudget, nullptr);
}

// ---------------------------------------------------------------------------
// MMA issuer (warp 1, one lane).  PASS 1: D[row, key] for the one or two 128-row
// M-tiles of the Q block.  PASS 2: D[key, row], N = n_cols rows.
// ---------------------------------------------------------------------------
template <int D, int PASS>
__device__ void issue(uint32_t tmem, unsigned char *sQ, unsigned char *sK, const Bars &B,
                      const int *ids, const Sched &S, volatile int *abort_flag) {
  using Gm = Geo<D>;
  // Operand descriptors: built once and stepped by constant offsets (the start
  // address field holds addr >> 4; shared memory stays below 2^18 bytes, so a
  // step never carries out of it).  The issuing thread shares its SMSP with busy
  // epilogue warps, so every instruction saved here keeps the tensor pipe fed.
  const uint64_t qd0 = tc::sdesc_sw128(tc::smem_u32(sQ));
  const uint64_t kd_base = tc::sdesc_sw128(tc::smem_u32(sK));
  const uint32_t idesc = PASS == 1 ? tc::idesc_bf16(128, KT) : tc::idesc_bf16(128, S.n_cols);
  uint32_t kt = 0, qv = 0;
  int prev_g = -1;
  bool ok = true;
  for (uint32_t it = 0; ok; ++it) {
    const int slot = it % IRING;
    if (!tc::mbar_wait(B.ifull + slot, (it / IRING) & 1, kWaitBudget, abort_flag)) {
      set_abort(abort_flag, S.status);
      break;
    }
    const int i = ids[slot];
    tc::mbar_arrive(B.iempty + slot);
    if (i < 0) break;
    Item w;
    Grp grp;
    item_of(S, i, w, grp);
    if (w.g != prev_g) {
      prev_g = w.g;
      if (qv > 0) tc::umma_commit(B.qempty);  // the previous Q block is free once these MMAs finish
      if (!tc::mbar_wait(B.qfull, qv & 1, kWaitBudget, abort_flag)) {
        set_abort(abort_flag, S.status);
        break;
      }
      ++qv;
      tc::fence_after_sync();
    }
    const bool two_mt = grp.nrows > 128;
    for (int j0 = w.j0; j0 < w.j1; j0 += KT, ++kt) {
      const int st = kt % STAGES;
      const uint32_t use = kt / STAGES;
      const int slot = kt & 1;
      const uint32_t tuse = kt >> 1;
      if (!tc::mbar_wait(B.full + st, use & 1, kWaitBudget, abort_flag) ||
          !tc::mbar_wait(B.tempty + slot, (tuse & 1) ^ 1, kWaitBudget, abort_flag)) {
        set_abort(abort_flag, S.status);
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint64_t kd0 = kd_base + (uint64_t)((st * Gm::KBYTES) >> 4);
      const uint32_t d0 = tmem + slot * 256;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t kd = kd0 + (uint64_t)(((kk / 4) * Gm::KSUB + (kk % 4) * 32) >> 4);
        const uint64_t qd = qd0 + (uint64_t)(((kk / 4) * Gm::QSUB + (kk % 4) * 32) >> 4);
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
  }
  // every MMA issued above completes before TMEM can be released
  tc::umma_commit(B.drain);
  tc::mbar_wait(B.drain, 0, kDrainBudget, nullptr);
}

// Sums above this force the exact-max path of the statistics epilogue: every
// term is then at most 2^64, so the running normaliser cannot overflow.
constexpr float kLazyLimit = 1.8446744e19f;

// sum_c 2^(x_c * c_log2 - m) over N logits, two at a time with packed fp32 math.
template <int N>
__device__ __forceinline__ float chunk_sum(const uint32_t *r, float c_log2, float m) {
  const float2 c2 = make_float2(c_log2, c_log2);
  const float2 nm2 = make_float2(-m, -m);
  float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < N; c += 4) {
    const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), c2, nm2);
    const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(r[c + 2]), __uint_as_float(r[c + 3])), c2, nm2);
    a0 = __fadd2_rn(a0, make_float2(tc::ex2(x0.x), tc::ex2(x0.y)));
    a1 = __fadd2_rn(a1, make_float2(tc::ex2(x1.x), tc::ex2(x1.y)));
  }
  const float2 a = __fadd2_rn(a0, a1);
  return a.x + a.y;
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

// The epilogue's next item: its leader (epilogue thread 0) takes it from the
// item ring and broadcasts it, so that all epilogue threads walk the same items
// and meet at the same named barriers.  -1: no item left (or aborting).
__device__ __forceinline__ int epi_next_item(uint32_t it, int et, const Bars &B, const int *ids,
                                             volatile int *bcast, volatile int *abort_flag,
                                             int *status) {
  if (et == 0) {
    const int slot = it % IRING;
    int i = -1;
    if (tc::mbar_wait(B.ifull + slot, (it / IRING) & 1, kWaitBudget, abort_flag))
      i = ids[slot];
    else
      set_abort(abort_flag, status);
    tc::mbar_arrive(B.iempty + slot);
    bcast[it & 1] = i;
  }
  tc::named_bar_sync(1, EPI_THREADS);
  return bcast[it & 1];
}

// ---------------------------------------------------------------------------
// The two passes.
// ---------------------------------------------------------------------------
template <int D, int PASS>
__global__ void __launch_bounds__(NT, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ Sched S) {
  using Gm = Geo<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = align1024(smem_raw);
  unsigned char *sQ = sm;
  unsigned char *sK = sm + Gm::QBYTES;
  const Bars B = carve_bars(sm + Gm::BAR_OFF);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Gm::MISC_OFF);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *ids = reinterpret_cast<int *>(sm + Gm::MISC_OFF + 16);                        // [IRING]
  volatile int *bcast = reinterpret_cast<volatile int *>(sm + Gm::MISC_OFF + 16 + 4 * IRING);  // [2]
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
    if (lane == 0) produce<D>(&tmQ, &tmK, sQ, sK, B, ids, S, abort_flag);
  } else if (warp == 1) {
    if (lane == 0) issue<D, PASS>(tmem, sQ, sK, B, ids, S, abort_flag);
  } else if (PASS == 1) {
    // ---- statistics: per-row running max and normaliser over each split ----
    const int ew = warp - 2;                // 0 .. EPI_WARPS-1
    const int wg = ew >> 2;                 // warpgroup 0..3
    const int mt = wg >> 1;                 // M-tile (rows 0..127 or 128..255 of the block)
    const int chalf = wg & 1;               // which 64 keys of each 128-key tile
    const int quarter = warp & 3;           // TMEM lane quarter this warp may access
    const int rit = quarter * 32 + lane;    // row within the M-tile
    const int rib = mt * 128 + rit;         // row within the block
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    float2 *xch = reinterpret_cast<float2 *>(sm + Gm::RED_OFF);  // [2 items][QROWS]
    uint32_t kt = 0;
    bool ok = true;
    int it = 0;
    // A warp that gives up keeps walking the same items and tiles (without
    // touching TMEM) so that every named barrier is reached by all epilogue threads.
    const int et = threadIdx.x - 64;
    for (uint32_t itn = 0;; ++itn) {
      const int i = epi_next_item(itn, et, B, ids, bcast, abort_flag, S.status);
      if (i < 0) break;
      Item w;
      Grp grp;
      item_of(S, i, w, grp);
      const bool has_mt = mt * 128 < grp.nrows;
      const int row = grp.r0 + rib;
      const int p_row = S.T - S.W + (row % S.W);
      const int jlim = min(w.j1, p_row + 1);  // keys this row may see in the split
      // where this row's (max, sum) over the split goes (only one thread per row writes)
      float2 *const pdst = (chalf == 0 && has_mt && rib < grp.nrows)
                               ? S.part + ((long long)w.g * S.ns + w.ks) * QROWS + rib
                               : nullptr;
      float m = -INFINITY, z = 0.f;
      for (int j0 = w.j0; j0 < w.j1; j0 += KT, ++kt) {
        const int slot = kt & 1;
        const uint32_t tuse = kt >> 1;
        if (ok && !tc::mbar_wait(B.tfull + slot, tuse & 1, kWaitBudget, abort_flag)) {
          set_abort(abort_flag, S.status);
          ok = false;
        }
        if (!ok) continue;
        tc::fence_after_sync();
        if (has_mt) {
          uint32_t r[64];
          const uint32_t col = tmem + lane_addr + slot * 256 + mt * 128 + chalf * 64;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            tc::tmem_ld16(col + q * 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16 * q]));
          tc::tmem_ld_wait();
          // fold the 64 logits of keys jb .. jb+63 (those below jlim are visible to
          // the row) into the row's running reference m and normaliser z
          const int jb = j0 + chalf * 64;
          if (jb + 64 <= jlim) {
            // every key visible: sum against the running reference m; only a sum
            // large enough to risk overflow (or the first chunk, m = -inf) takes
            // the exact-max path (inline: out of line measured 8% slower)
            float sum = chunk_sum<64>(r, S.c_log2, m);
            if (!(sum <= kLazyLimit)) {
              float cm = -INFINITY;
#pragma unroll
              for (int c = 0; c < 64; ++c) cm = fmaxf(cm, __uint_as_float(r[c]));
              const float mnew = fmaxf(m, cm * S.c_log2);
              sum = chunk_sum<64>(r, S.c_log2, mnew);
              z = z * tc::ex2(m - mnew);
              m = mnew;
            }
            z += sum;
          } else if (jb < jlim) {
            float cm = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (jb + c < jlim) cm = fmaxf(cm, __uint_as_float(r[c]));
            const float mnew = fmaxf(m, cm * S.c_log2);
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              const float e = tc::ex2(fmaf(__uint_as_float(r[c]), S.c_log2, -mnew));
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
      float2 *xb = xch + (it & 1) * QROWS;
      if (chalf == 1) xb[rib] = make_float2(m, z);
      tc::named_bar_sync(1, EPI_THREADS);
      if (ok && pdst) {
        const float2 o = xb[rib];
        const float M = fmaxf(m, o.x);
        float Z = 0.f;
        if (m != -INFINITY) Z += z * tc::ex2(m - M);
        if (o.x != -INFINITY) Z += o.y * tc::ex2(o.x - M);
        *pdst = make_float2(M, Z);
      }
      ++it;
    }
  } else {
    // ---- column mass: per key, the block rows' probability mass ----
    const int et = threadIdx.x - 64;        // 0 .. EPI_THREADS-1
    const int ew = warp - 2;
    const int wg = ew >> 2;                 // this warpgroup takes column chunks wg, wg+4, ...
    const int quarter = warp & 3;
    const int key_in_tile = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const int n_chunks = S.n_cols / 16;
    float *sM = reinterpret_cast<float *>(sm + Gm::STAT_OFF);
    int *sPos = reinterpret_cast<int *>(sM + QROWS);
    float *sRed = reinterpret_cast<float *>(sm + Gm::RED_OFF);
    uint32_t kt = 0;
    bool ok = true;
    int prev_g = -1;
    // A warp that gives up keeps walking the same items and tiles (without
    // touching TMEM) so that every named barrier below is reached by all 512
    // epilogue threads.
    for (uint32_t itn = 0;; ++itn) {
      const int i = epi_next_item(itn, et, B, ids, bcast, abort_flag, S.status);
      if (i < 0) break;
      Item w;
      Grp grp;
      item_of(S, i, w, grp);
      if (w.g != prev_g) {
        prev_g = w.g;  // the previous block's readers passed the item barrier
        for (int r = et; r < QROWS; r += EPI_THREADS) {
          if (r < grp.nrows) {
            sM[r] = S.fin[(long long)w.g * QROWS + r];
            sPos[r] = S.T - S.W + ((grp.r0 + r) % S.W);
          } else {
            sM[r] = -INFINITY;  // padding rows contribute 2^-inf = 0
            sPos[r] = -1;
          }
        }
        tc::named_bar_sync(1, EPI_THREADS);
      }
      float *dst = S.nrb == 1 ? S.s_out + (long long)grp.u * S.T
                              : S.pcol + ((long long)grp.u * S.nrb + grp.rb) * S.T;
      for (int j0 = w.j0; j0 < w.j1; j0 += KT, ++kt) {
        const int slot = kt & 1;
        const uint32_t tuse = kt >> 1;
        if (ok && !tc::mbar_wait(B.tfull + slot, tuse & 1, kWaitBudget, abort_flag)) {
          set_abort(abort_flag, S.status);
          ok = false;
        }
        const int j = j0 + key_in_tile;
        float acc = 0.f;
        if (ok) {
          tc::fence_after_sync();
          const bool masked = j0 + KT > grp.kfull;
          float2 acc2 = make_float2(0.f, 0.f);
          const float2 c2 = make_float2(S.c_log2, S.c_log2);
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
        // add the four warpgroups' shares (fixed order) and store the key's mass.
        // Only the four warps on the same TMEM lane quarter (the same 32 keys)
        // exchange, so they meet at their quarter's own barrier; the exchange
        // buffer alternates between tiles, so one barrier per tile suffices
        float *red = sRed + (kt & 1) * 4 * KT;
        if (wg > 0) red[wg * KT + key_in_tile] = acc;
        tc::named_bar_sync(2 + quarter, 4 * 32);
        if (ok && wg == 0 && j < w.j1)
          dst[j] = acc + (red[KT + key_in_tile] + red[2 * KT + key_in_tile] + red[3 * KT + key_in_tile]);
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

// fin[g][r] = -(M + log2 Z) of row r of block g over the block's splits, in
// split order (-inf for the padding rows of a partial block).
__global__ void score_merge_kernel(const float2 *__restrict__ part, int T, int W, int gw, int nrb,
                                   int ns, int split_len, long long total, float *__restrict__ fin) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int g = static_cast<int>(i / QROWS);
  const int r = static_cast<int>(i % QROWS);
  const Grp grp = group_of(g, T, W, gw, nrb, split_len);
  if (r >= grp.nrows) {
    fin[i] = -INFINITY;
    return;
  }
  const float2 *p = part + (long long)g * ns * QROWS + r;
  float M = -INFINITY;
  for (int s = 0; s < grp.nsplit; ++s) M = fmaxf(M, p[(long long)s * QROWS].x);
  float Z = 0.f;
  for (int s = 0; s < grp.nsplit; ++s) {
    const float2 v = p[(long long)s * QROWS];
    if (v.x != -INFINITY) Z += v.y * exp2f(v.x - M);
  }
  // 2^(x c - M) / Z = 2^(x c - (M + log2 Z)); every row sees key 0, so Z >= 1
  fin[i] = -(M + log2f(Z));
}

// s[u][j] = sum over the row blocks that see key j of their column sums, in block order.
__global__ void score_block_sum_kernel(const float *__restrict__ pcol, int T, int W, int gw, int nrb,
                                       int split_len, long long total, float *__restrict__ s) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int u = static_cast<int>(idx / T);
  const int j = static_cast<int>(idx % T);
  float acc = 0.f;
  for (int rb = 0; rb < nrb; ++rb) {
    const Grp grp = group_of(u * nrb + rb, T, W, gw, nrb, split_len);
    if (j < grp.kend) acc += __ldg(pcol + ((long long)u * nrb + rb) * T + j);
  }
  s[idx] = acc;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// rows x d bf16 matrix, boxes of 64 elements x 128 rows, 128-byte swizzle.
bool encode_rows(CUtensorMap *map, const void *base, long rows, int d) {
  return tc::encode_rows_sw128(map, base, rows, d, 2, 128);
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <int D>
int run_tc(const void *Q, const void *K, int B, int Hq, int Hkv, int T, int W, float scale,
           float *s, void *ws, const ScorePlan &plan, int *status, cudaStream_t st) {
  using Gm = Geo<D>;
  const long long units = (long long)B * Hkv;
  const TcLayout L = tc_layout(B, Hq, Hkv, T, W);
  unsigned char *base = static_cast<unsigned char *>(ws);
  Sched S;
  S.T = T;
  S.W = W;
  S.G = Hq / Hkv;
  S.Hq = Hq;
  S.Hkv = Hkv;
  S.gw = plan.gw;
  S.nrb = L.nrb;
  S.ns = L.ns;
  S.split_len = L.split_len;
  S.n_cols = L.nrb > 1 ? QROWS : ((plan.gw + 15) / 16) * 16;
  if (units * L.nrb * L.ns > 0x7FFFFFFFLL || units * L.nrb > 0x7FFFFFFFLL / QROWS) return KV_ERR_UNSUPPORTED;
  S.n_items = static_cast<int>(units * L.nrb * L.ns);
  S.n_groups = static_cast<int>(units * L.nrb);
  unsigned *next = reinterpret_cast<unsigned *>(base + L.ctrl_off);  // one claim counter per pass
  S.c_log2 = scale * 1.4426950408889634f;
  S.part = reinterpret_cast<float2 *>(base + L.part_off);
  float *fin = reinterpret_cast<float *>(base + L.fin_off);
  S.fin = fin;
  S.pcol = L.nrb > 1 ? reinterpret_cast<float *>(base + L.pcol_off) : nullptr;
  S.s_out = s;
  S.status = status;

  CUtensorMap tmQ, tmK;
  if (!encode_rows(&tmQ, Q, (long)B * Hq * W, D) || !encode_rows(&tmK, K, units * T, D))
    return KV_ERR_CUDA;
  if (ensure_smem((const void *)score_tc_kernel<D, 1>, Gm::SMEM) ||
      ensure_smem((const void *)score_tc_kernel<D, 2>, Gm::SMEM))
    return KV_ERR_CUDA;
  const int sms = device_sm_count();
  const unsigned grid = (unsigned)(S.n_items < sms ? S.n_items : sms);
  const cudaError_t e = cudaMemsetAsync(next, 0, 2 * sizeof(unsigned), st);
  if (e != cudaSuccess) return cuda_failure(e, "scoring: clearing the claim counters");
  S.next = next;
  score_tc_kernel<D, 1><<<grid, NT, Gm::SMEM, st>>>(tmQ, tmK, S);
  const long long rows = units * L.nrb * QROWS;
  score_merge_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, st>>>(
      S.part, T, W, plan.gw, L.nrb, L.ns, L.split_len, rows, fin);
  S.next = next + 1;
  score_tc_kernel<D, 2><<<grid, NT, Gm::SMEM, st>>>(tmQ, tmK, S);
  int launches = 3;
  if (L.nrb > 1) {
    const long long total = units * T;
    score_block_sum_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(
        S.pcol, T, W, plan.gw, L.nrb, L.split_len, total, s);
    ++launches;
  }
  return launch_status(launches);
}

}  // namespace

// Workspace layout and work split of the tensor-core path (shared with plan_score).
TcLayout tc_layout(int B, int Hq, int Hkv, int T, int W) {
  TcLayout L{};
  const long long units = (long long)B * Hkv;
  const int gw = (Hq / Hkv) * W;
  L.nrb = (gw + QROWS - 1) / QROWS;
  const int tiles = (T + KT - 1) / KT;
  int per;  // tiles per split
  if (L.nrb == 1) {
    // about 16 items per SM keeps the round-robin tail short
    long long want = (16LL * kNumSmsHint + units - 1) / (units > 0 ? units : 1);
    if (want < 1) want = 1;
    if (want > tiles) want = tiles;
    per = (int)((tiles + want - 1) / want);
    if (per < 4) per = 4;  // an item reloads its Q block: keep a few tiles per item
  } else {
    per = tiles;  // row blocks already give many items; the claims balance their sizes
  }
  if (per > tiles) per = tiles;
  L.split_len = per * KT;
  L.ns = (T + L.split_len - 1) / L.split_len;
  const long long groups = units * L.nrb;
  L.ctrl_off = 0;
  L.part_off = 256;
  L.fin_off = L.part_off + align256(sizeof(float2) * (size_t)groups * L.ns * QROWS);
  L.pcol_off = L.fin_off + align256(sizeof(float) * (size_t)groups * QROWS);
  L.bytes = L.pcol_off + (L.nrb > 1 ? align256(sizeof(float) * (size_t)groups * T) : 0);
  return L;
}

bool score_tc_eligible(int dtype, int d, int Hq, int Hkv, int W) {
  (void)Hq;
  (void)Hkv;
  (void)W;
  return dtype == KV_BF16 && (d == 64 || d == 128);
}

int launch_score_obs_tc(const void *Q, const void *K, int B, int Hq, int Hkv, int T, int d, int W,
                        float scale, float *s, void *ws, const ScorePlan &plan, int *status,
                        cudaStream_t st) {
  if (d == 128) return run_tc<128>(Q, K, B, Hq, Hkv, T, W, scale, s, ws, plan, status, st);
  return run_tc<64>(Q, K, B, Hq, Hkv, T, W, scale, s, ws, plan, status, st);
}

}  // namespace kvc
