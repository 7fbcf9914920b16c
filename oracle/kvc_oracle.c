/*
 * kvc_oracle.c -- plain, slow, float64 CPU oracle of the KV-cache eviction path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or helper with the CUDA library; it
 * reads the same input bytes (bf16 bit patterns or float32) and computes every
 * quantity in double precision, one obvious loop at a time, in the order the
 * pages describe.  Independent (batch, head) units may run on OpenMP threads;
 * nothing inside a unit is blocked, fused or reordered.
 *
 * Sources (page title, section):
 *   [H2O]    "H2O 完全拆解：抓住 KV Cache 里的「重击者」，20% 预算无损生成（NeurIPS 2023）"
 *            sections 观察二 (accumulated attention o_s), 问题形式化 (|S_i| = k,
 *            at most one eviction per step, renormalised restricted attention),
 *            贪心驱逐算法 (Algorithm 1), 为什么是「重击者 + 最近」双缓冲,
 *            为什么要按头独立驱逐, FlexGen 改造：预分配 + 原地覆写,
 *            两套代码：模拟版与真实丢弃版.
 *   [HubKV]  "HubKV walkthrough", sections 核心概念：Modular vs. Submodular,
 *            Theory Lens (SMD discount), 局部理论保证 (bounded perturbation),
 *            Method: 最终算法：四步修正原始分数 (local hubs, SMD discount,
 *            head calibration, ratio gate).
 *   [KVblog] KV-cache survey blog, §1.1 (scaled dot-product attention with
 *            1/sqrt(d_head)), §1.3 (KV-cache size), §3.3 (GQA), §4.3 (SnapKV
 *            prefill observation window), §4.4 (PyramidKV per-layer budgets).
 *   [NestedKV] "Technische Samenvatting: NestedKV", sections 1. Continuum
 *            Geheugentoestand (three key anchors, cosine anomaly scores),
 *            2. Buitenste Leraar (head-adaptive blending, surprise routing),
 *            3. Hoofd-gewijze Geheugentoewijzing (competitive head-wise budget).
 *
 * Readings taken where the pages are silent (each one is listed in the design
 * notes as well):
 *   - observation window = the last W prompt positions as queries, causal over
 *     keys at or before each query's own position ([KVblog] §4.3);
 *   - column mass is a SUM over window rows and over the G query heads of a GQA
 *     group ([H2O] 观察二 "accumulated");
 *   - the gate's q_i is the SMD-discounted score; selectivity is one minus the
 *     normalised entropy of the head's score distribution ("parity unpinned"
 *     beyond the clip range, monotonicity and the identical-heads case);
 *   - Top-K order is (z descending, position ascending); the decode victim is
 *     (accumulator ascending, position ascending), i.e. the oldest on ties.
 *
 * dtype codes: 0 = bf16 (uint16 bit patterns), 1 = float32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_BF16 0
#define OR_F32 1
#define OR_FLAG_ALG1 1
#define OR_HUB_AVGPOOL 1    /* hubkv_refine variant: average-pool smoothing instead of hubs */
#define OR_HUB_FIXED_HEAD 2 /* hubkv_refine variant: fixed head weight (beta = 1) */

/* Read element i of a bf16 or f32 array as a double. bf16 is the upper half of
 * an IEEE float32, so the value is exact. */
static double or_load(const void *base, size_t i, int dtype) {
  if (dtype == OR_BF16) {
    uint16_t bits = ((const uint16_t *)base)[i];
    uint32_t wide = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &wide, sizeof f);
    return (double)f;
  }
  return (double)((const float *)base)[i];
}

static size_t or_elem_bytes(int dtype) { return dtype == OR_BF16 ? 2u : 4u; }

static int or_is_finite(double x) { return x == x && x - x == 0.0; }

/* KV-cache size in bytes: 2 (K and V) x layers x KV heads x d_head x tokens x
 * bytes per element ([KVblog] §1.3). */
long long oracle_kv_cache_bytes(long long L, long long Hkv, long long d, long long T,
                                long long elem_bytes) {
  return 2LL * L * Hkv * d * T * elem_bytes;
}

/* ---------------------------------------------------------------------------
 * Step 1: observation-window scoring.
 *
 * For unit (b, h) with KV head h serving query heads h*G .. h*G+G-1:
 *   for each such query head g and window row w (prompt position p = T-W+w):
 *     l_j = scale * <q_{g,w}, k_j>           for j = 0..p      ([KVblog] §1.1)
 *     P_j = exp(l_j - max l) / sum_t exp(l_t - max l)
 *     s_j += P_j                                                 ([H2O] 观察二)
 * Keys after a row's own position receive nothing from that row.
 * Layouts: Q [B][Hq][W][d], K [B][Hkv][T][d], s [B][Hkv][T].
 * Returns 0, or -1 on bad arguments or non-finite input.
 * ------------------------------------------------------------------------- */
int oracle_score_obs(const void *Q, const void *K, int B, int Hq, int Hkv, int T, int d,
                     int W, double scale, int dtype, double *s_out) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || T <= 0 || d <= 0 || W <= 0 ||
      W > T)
    return -1;
  const int G = Hq / Hkv;
  const long long units = (long long)B * Hkv;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (long long u = 0; u < units; ++u) {
    const int b = (int)(u / Hkv), h = (int)(u % Hkv);
    double *s = s_out + u * (long long)T;
    double *logit = (double *)malloc(sizeof(double) * (size_t)T);
    if (!logit) {
      bad = 1;
      continue;
    }
    for (int j = 0; j < T; ++j) s[j] = 0.0;
    for (int g = 0; g < G; ++g) {
      const int hq = h * G + g;
      for (int w = 0; w < W; ++w) {
        const int p = T - W + w;
        const size_t qoff = (((size_t)b * Hq + hq) * W + w) * (size_t)d;
        double m = -INFINITY;
        for (int j = 0; j <= p; ++j) {
          const size_t koff = (((size_t)b * Hkv + h) * T + j) * (size_t)d;
          double dot = 0.0;
          for (int c = 0; c < d; ++c) dot += or_load(Q, qoff + c, dtype) * or_load(K, koff + c, dtype);
          logit[j] = scale * dot;
          if (!or_is_finite(logit[j])) bad = 1;
          if (logit[j] > m) m = logit[j];
        }
        double Z = 0.0;
        for (int j = 0; j <= p; ++j) Z += exp(logit[j] - m);
        for (int j = 0; j <= p; ++j) s[j] += exp(logit[j] - m) / Z;
      }
    }
    free(logit);
  }
  return bad ? -1 : 0;
}

/* ---------------------------------------------------------------------------
 * Step 2: HubKV refinement ([HubKV] Method, four steps).
 *
 *   1. local hubs: M_i = max of s over |j - i| <= pool_width/2 (window cut at the
 *      sequence ends); i is a hub iff s_i == M_i;
 *   2. SMD discount: q_i = s_i for hubs, gamma * s_i otherwise;
 *   3. head calibration: sel_h = 1 - H_h / ln T with H_h the entropy of the
 *      head's normalised scores (0 ln 0 = 0; T = 1 or an all-zero head gives
 *      sel = 0); beta_h = clip(sel_h / mean over the unit's heads, lo, hi), or 1
 *      when that mean is 0.  The unit is one batch row: heads b*H .. b*H+H-1;
 *   4. ratio gate: z_i = s_i + r^2 (beta_h q_i - s_i).
 * s, z [B][H][T]; beta, sel [B][H] (either may be NULL).
 *
 * Variants the HubKV page reports as weaker (尝试路线：效果一般的可能原因), as
 * flags: OR_HUB_AVGPOOL replaces steps 1-2 by average-pool smoothing, q_i = the
 * mean of s over the same window ("CommunitySmooth"); OR_HUB_FIXED_HEAD replaces
 * step 3 by a fixed head weight, beta_h = 1.
 * ------------------------------------------------------------------------- */
int oracle_hubkv_refine_ex(const double *s, int B, int H, int T, int pool_width, double gamma,
                           double r, double beta_lo, double beta_hi, int flags, double *z_out,
                           double *beta_out, double *sel_out) {
  if (B < 0 || H <= 0 || T <= 0 || pool_width <= 0 || pool_width % 2 == 0 ||
      beta_lo > beta_hi || (flags & ~(OR_HUB_AVGPOOL | OR_HUB_FIXED_HEAD)))
    return -1;
  const int half = pool_width / 2;
  double *sel = (double *)malloc(sizeof(double) * (size_t)(B > 0 ? B : 1) * H);
  if (!sel) return -1;
  for (long long u = 0; u < (long long)B * H; ++u) {
    const double *sv = s + u * (long long)T;
    double S = 0.0;
    for (int i = 0; i < T; ++i) S += sv[i];
    double ent = 0.0;
    if (S > 0.0) {
      for (int i = 0; i < T; ++i) {
        const double p = sv[i] / S;
        if (p > 0.0) ent -= p * log(p);
      }
    }
    sel[u] = (T > 1 && S > 0.0) ? 1.0 - ent / log((double)T) : 0.0;
    if (sel_out) sel_out[u] = sel[u];
  }
  for (int b = 0; b < B; ++b) {
    double mean = 0.0;
    for (int h = 0; h < H; ++h) mean += sel[(long long)b * H + h];
    mean /= (double)H;
    for (int h = 0; h < H; ++h) {
      const long long u = (long long)b * H + h;
      double beta = 1.0;
      if (mean != 0.0 && !(flags & OR_HUB_FIXED_HEAD)) {
        beta = sel[u] / mean;
        if (beta < beta_lo) beta = beta_lo;
        if (beta > beta_hi) beta = beta_hi;
      }
      if (beta_out) beta_out[u] = beta;
      const double *sv = s + u * (long long)T;
      double *zv = z_out + u * (long long)T;
      for (int i = 0; i < T; ++i) {
        double qi;
        if (flags & OR_HUB_AVGPOOL) {
          /* the smoothing variant: the mean of s over the window (cut at the ends) */
          double sum = 0.0;
          int cnt = 0;
          for (int j = i - half; j <= i + half; ++j)
            if (j >= 0 && j < T) {
              sum += sv[j];
              ++cnt;
            }
          qi = sum / cnt;
        } else {
          double M = -INFINITY;
          for (int j = i - half; j <= i + half; ++j)
            if (j >= 0 && j < T && sv[j] > M) M = sv[j];
          qi = (sv[i] == M) ? sv[i] : gamma * sv[i];
        }
        zv[i] = sv[i] + r * r * (beta * qi - sv[i]);
      }
    }
  }
  free(sel);
  return 0;
}

int oracle_hubkv_refine(const double *s, int B, int H, int T, int pool_width, double gamma,
                        double r, double beta_lo, double beta_hi, double *z_out,
                        double *beta_out, double *sel_out) {
  return oracle_hubkv_refine_ex(s, B, H, T, pool_width, gamma, r, beta_lo, beta_hi, 0, z_out,
                                beta_out, sel_out);
}

/* ---------------------------------------------------------------------------
 * Step 3: budgeted per-head Top-K with a protected recent window.
 * Keep the last R positions [T-R, T) unconditionally ([H2O] 双缓冲), and the
 * k-R best of [0, T-R) ordered by (z descending, position ascending).  Output
 * the k kept positions in ascending order.  Each head selects on its own
 * ([H2O] 按头独立驱逐).  z [B][H][T], idx [B][H][k].  Requires 0 <= R < k <= T.
 * With S sink positions ([KVblog] §4.1-4.2: the first few tokens are kept as
 * attention sinks) the first S positions are kept too and the heavy part is the
 * k-R-S best of [S, T-R); requires S + R < k.
 * ------------------------------------------------------------------------- */
typedef struct {
  double z;
  int pos;
} or_cand;

static int or_cmp_desc(const void *a, const void *b) {
  const or_cand *x = (const or_cand *)a, *y = (const or_cand *)b;
  if (x->z > y->z) return -1;
  if (x->z < y->z) return 1;
  return (x->pos > y->pos) - (x->pos < y->pos);
}

static int or_cmp_int(const void *a, const void *b) {
  const int x = *(const int *)a, y = *(const int *)b;
  return (x > y) - (x < y);
}

int oracle_select_topk_ex(const double *z, int B, int H, int T, int k, int recent, int sink,
                          int32_t *idx_out) {
  if (B < 0 || H <= 0 || T <= 0 || recent < 0 || sink < 0 || k <= recent + sink || k > T)
    return -1;
  const int n = T - recent - sink, nh = k - recent - sink;
  or_cand *c = (or_cand *)malloc(sizeof(or_cand) * (size_t)(n > 0 ? n : 1));
  int *keep = (int *)malloc(sizeof(int) * (size_t)k);
  if (!c || !keep) {
    free(c);
    free(keep);
    return -1;
  }
  for (long long u = 0; u < (long long)B * H; ++u) {
    const double *zv = z + u * (long long)T;
    for (int i = 0; i < n; ++i) {
      c[i].z = zv[sink + i];
      c[i].pos = sink + i;
    }
    qsort(c, (size_t)n, sizeof(or_cand), or_cmp_desc);
    for (int m = 0; m < nh; ++m) keep[m] = c[m].pos;
    for (int m = 0; m < recent; ++m) keep[nh + m] = T - recent + m;
    for (int m = 0; m < sink; ++m) keep[nh + recent + m] = m;
    qsort(keep, (size_t)k, sizeof(int), or_cmp_int);
    for (int m = 0; m < k; ++m) idx_out[u * (long long)k + m] = keep[m];
  }
  free(c);
  free(keep);
  return 0;
}

int oracle_select_topk(const double *z, int B, int H, int T, int k, int recent,
                       int32_t *idx_out) {
  return oracle_select_topk_ex(z, B, H, T, k, recent, 0, idx_out);
}

/* ---------------------------------------------------------------------------
 * Step 4: gather-compaction ("real drop", [H2O] 两套代码).
 *   K_out[m] = K[idx[m]], V_out[m] = V[idx[m]], pos[m] = idx[m],
 *   acc[m] = s[idx[m]] (the attention mass received so far), len = k.
 * K, V [B][H][T][d]; K_out, V_out [B][H][cap][d]; pos, acc [B][H][cap];
 * len [B][H].  Slots k..cap-1 are left untouched.  s and acc may be NULL.
 * ------------------------------------------------------------------------- */
int oracle_compact(const void *K, const void *V, const double *s, const int32_t *idx,
                   int B, int H, int T, int k, int d, int dtype, void *K_out, void *V_out,
                   int cap, int32_t *pos_out, float *acc_out, int32_t *len_out) {
  if (B < 0 || H <= 0 || T <= 0 || k <= 0 || k > T || d <= 0 || cap < k) return -1;
  const size_t row = (size_t)d * or_elem_bytes(dtype);
  for (long long u = 0; u < (long long)B * H; ++u) {
    for (int m = 0; m < k; ++m) {
      const int j = idx[u * k + m];
      if (j < 0 || j >= T) return -1;
      memcpy((char *)K_out + ((size_t)u * cap + m) * row, (const char *)K + ((size_t)u * T + j) * row, row);
      memcpy((char *)V_out + ((size_t)u * cap + m) * row, (const char *)V + ((size_t)u * T + j) * row, row);
      pos_out[u * (long long)cap + m] = j;
      if (s && acc_out) acc_out[u * (long long)cap + m] = (float)s[u * (long long)T + j];
    }
    len_out[u] = k;
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Layer-level competitive budget ([NestedKV] 3. Hoofd-gewijze
 * Geheugentoewijzing: the (token, head) pairs with the highest scores across
 * the layer win, subject to a per-head minimum; [KVblog] §4.4 PyramidKV: the
 * budget belongs to the layer rather than to each head).
 * Batch row b is one layer; its H heads share `budget` kept positions:
 *   1. every head keeps its sinks [0, sink) and its recent window [T-recent, T);
 *   2. floor: every head keeps its floor - sink - recent best positions of
 *      [sink, T-recent) in the order (z descending, position ascending), so that
 *      each head keeps at least `floor` positions;
 *   3. competition: the budget - H*floor slots left go to the best of the row's
 *      (head, position) pairs with position in [sink, T-recent) not kept yet, in
 *      the order (z descending, head ascending, position ascending).
 * Output, CSR: head h of row b kept positions idx[b][off[b][h] .. off[b][h+1]-1]
 * in ascending order; off[b][0] = 0 and off[b][H] = budget.
 * Steps 2-3 give the largest score sum over all sets that keep the protected
 * positions, at least `floor` per head and `budget` in all.
 * z [B][H][T]; idx [B][budget]; off [B][H+1].
 * ------------------------------------------------------------------------- */
typedef struct {
  double z;
  int head;
  int pos;
} or_pair;

static int or_cmp_pair_desc(const void *a, const void *b) {
  const or_pair *x = (const or_pair *)a, *y = (const or_pair *)b;
  if (x->z > y->z) return -1;
  if (x->z < y->z) return 1;
  if (x->head != y->head) return (x->head > y->head) - (x->head < y->head);
  return (x->pos > y->pos) - (x->pos < y->pos);
}

int oracle_select_budget(const double *z, int B, int H, int T, int budget, int floor_k,
                         int recent, int sink, int32_t *idx_out, int32_t *off_out) {
  if (B < 0 || H <= 0 || T <= 0 || recent < 0 || sink < 0 || floor_k < 1 ||
      floor_k < recent + sink || floor_k > T || budget < (long long)H * floor_k ||
      budget > (long long)H * T)
    return -1;
  const int n = T - recent - sink, nf = floor_k - recent - sink;
  or_cand *c = (or_cand *)malloc(sizeof(or_cand) * (size_t)(n > 0 ? n : 1));
  or_pair *pool = (or_pair *)malloc(sizeof(or_pair) * (size_t)H * (size_t)(n > 0 ? n : 1));
  unsigned char *kept = (unsigned char *)malloc((size_t)H * (size_t)T);
  if (!c || !pool || !kept) {
    free(c);
    free(pool);
    free(kept);
    return -1;
  }
  for (int b = 0; b < B; ++b) {
    memset(kept, 0, (size_t)H * (size_t)T);
    long long np = 0;
    for (int h = 0; h < H; ++h) {
      const double *zv = z + ((long long)b * H + h) * T;
      unsigned char *kh = kept + (size_t)h * T;
      for (int m = 0; m < sink; ++m) kh[m] = 1;                  /* step 1 */
      for (int m = T - recent; m < T; ++m) kh[m] = 1;
      for (int i = 0; i < n; ++i) {
        c[i].z = zv[sink + i];
        c[i].pos = sink + i;
      }
      qsort(c, (size_t)n, sizeof(or_cand), or_cmp_desc);
      for (int m = 0; m < nf; ++m) kh[c[m].pos] = 1;             /* step 2 */
      for (int m = nf; m < n; ++m) {
        pool[np].z = c[m].z;
        pool[np].head = h;
        pool[np].pos = c[m].pos;
        ++np;
      }
    }
    qsort(pool, (size_t)np, sizeof(or_pair), or_cmp_pair_desc);
    const long long extra = (long long)budget - (long long)H * floor_k;
    for (long long m = 0; m < extra; ++m)                         /* step 3 */
      kept[(size_t)pool[m].head * T + pool[m].pos] = 1;
    int32_t *ib = idx_out + (long long)b * budget;
    int32_t *ob = off_out + (long long)b * (H + 1);
    int w = 0;
    for (int h = 0; h < H; ++h) {
      ob[h] = w;
      for (int p = 0; p < T; ++p)
        if (kept[(size_t)h * T + p]) ib[w++] = p;
    }
    ob[H] = w;
  }
  free(c);
  free(pool);
  free(kept);
  return 0;
}

/* ---------------------------------------------------------------------------
 * Ragged gather-compaction: Step 4 for the per-head counts that the layer
 * budget produces.  Head h of row b keeps n = off[b][h+1] - off[b][h] rows:
 *   K_out[m] = K[idx[off + m]], V_out[m] = V[idx[off + m]], pos[m] = idx[off + m],
 *   acc[m] = s[idx[off + m]], len = n, for m < n; slots n..cap-1 untouched.
 * K, V [B][H][T][d]; idx [B][budget]; off [B][H+1]; K_out, V_out [B][H][cap][d];
 * pos, acc [B][H][cap]; len [B][H].  Returns -1 when an offset or an index is out
 * of range or a head keeps more than cap rows.
 * ------------------------------------------------------------------------- */
int oracle_compact_ragged(const void *K, const void *V, const double *s, const int32_t *idx,
                          const int32_t *off, int B, int H, int T, int budget, int d, int dtype,
                          void *K_out, void *V_out, int cap, int32_t *pos_out, float *acc_out,
                          int32_t *len_out) {
  if (B < 0 || H <= 0 || T <= 0 || budget < 0 || d <= 0 || cap < 0) return -1;
  const size_t row = (size_t)d * or_elem_bytes(dtype);
  for (int b = 0; b < B; ++b) {
    const int32_t *ob = off + (long long)b * (H + 1);
    for (int h = 0; h < H; ++h) {
      const long long u = (long long)b * H + h;
      const int lo = ob[h], hi = ob[h + 1];
      if (lo < 0 || hi < lo || hi > budget || hi - lo > cap) return -1;
      for (int m = 0; m < hi - lo; ++m) {
        const int j = idx[(long long)b * budget + lo + m];
        if (j < 0 || j >= T) return -1;
        memcpy((char *)K_out + ((size_t)u * cap + m) * row, (const char *)K + ((size_t)u * T + j) * row, row);
        memcpy((char *)V_out + ((size_t)u * cap + m) * row, (const char *)V + ((size_t)u * T + j) * row, row);
        pos_out[u * cap + m] = j;
        if (s && acc_out) acc_out[u * cap + m] = (float)s[u * (long long)T + j];
      }
      len_out[u] = hi - lo;
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * NestedKV key-only scoring ([NestedKV] 1. Continuum Geheugentoestand and
 * 2. Buitenste Leraar).  Per unit (b, h), over the head's T keys:
 *   normalised keys   kh_i = k_i / |k_i|  (0 for a zero key);
 *   three anchors     mu_s    = mean of kh over all T keys (stable);
 *                     mu_e(i) = mean of kh over i's block, blocks of
 *                               blk = ceil(T / n_blocks) consecutive keys
 *                               (episodic; the last block may be shorter);
 *                     mu_c(i) = mean of kh over [max(0, i-window+1), i]
 *                               (current: causal moving mean, i included);
 *   anomaly scores    a_k(i) = -cos(kh_i, mu_k(i)), cos = 0 when a norm is 0;
 *   discriminative power per scale D_k = (mean of the n_disc largest a_k) -
 *                     (mean of the n_disc smallest a_k), over the head's tokens;
 *   scale weights     w = softmax over the three scales of D_k + log_prior[k];
 *   blend             a_blend(i) = sum_k w_k a_k(i);
 *   surprise          sigma(i) = population standard deviation of the three a_k(i);
 *   routing           score(i) = max_k a_k(i) if sigma(i) > thresh, else a_blend(i).
 * K [B][H][T][d]; score [B][H][T]; a_out [B][H][3][T] (s, e, c; may be NULL);
 * sigma_out [B][H][T] (may be NULL); w_out [B][H][3] (may be NULL).
 * ------------------------------------------------------------------------- */
static double or_cos(const double *x, const double *mu, int d) {
  double dot = 0.0, nx = 0.0, nm = 0.0;
  for (int f = 0; f < d; ++f) {
    dot += x[f] * mu[f];
    nx += x[f] * x[f];
    nm += mu[f] * mu[f];
  }
  if (nx == 0.0 || nm == 0.0) return 0.0;
  return dot / (sqrt(nx) * sqrt(nm));
}

static int or_cmp_double(const void *a, const void *b) {
  const double x = *(const double *)a, y = *(const double *)b;
  return (x > y) - (x < y);
}

int oracle_nested_score(const void *K, int B, int H, int T, int d, int dtype, int window,
                        int n_blocks, int n_disc, const double *log_prior, double thresh,
                        double *score_out, double *a_out, double *sigma_out, double *w_out) {
  if (B < 0 || H <= 0 || T <= 0 || d <= 0 || window < 1 || n_blocks < 1 || n_disc < 1 ||
      n_disc > T || !log_prior || !score_out)
    return -1;
  const int blk = (T + n_blocks - 1) / n_blocks;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (long long u = 0; u < (long long)B * H; ++u) {
    double *kh = (double *)malloc(sizeof(double) * (size_t)T * d);
    double *a = (double *)malloc(sizeof(double) * 3 * (size_t)T);
    double *srt = (double *)malloc(sizeof(double) * (size_t)T);
    double *mu = (double *)malloc(sizeof(double) * (size_t)d);
    if (!kh || !a || !srt || !mu) {
#pragma omp atomic write
      bad = 1;
      free(kh); free(a); free(srt); free(mu);
      continue;
    }
    /* normalised keys */
    for (int i = 0; i < T; ++i) {
      double nrm = 0.0;
      for (int f = 0; f < d; ++f) {
        const double v = or_load(K, ((size_t)u * T + i) * d + f, dtype);
        if (!or_is_finite(v)) {
#pragma omp atomic write
          bad = 1;
        }
        kh[(size_t)i * d + f] = v;
        nrm += v * v;
      }
      nrm = sqrt(nrm);
      for (int f = 0; f < d; ++f) kh[(size_t)i * d + f] = nrm > 0.0 ? kh[(size_t)i * d + f] / nrm : 0.0;
    }
    /* stable anchor */
    for (int f = 0; f < d; ++f) {
      double sum = 0.0;
      for (int j = 0; j < T; ++j) sum += kh[(size_t)j * d + f];
      mu[f] = sum / T;
    }
    for (int i = 0; i < T; ++i) a[i] = -or_cos(kh + (size_t)i * d, mu, d);
    /* episodic anchor, one block at a time */
    for (int lo = 0; lo < T; lo += blk) {
      const int hi = lo + blk < T ? lo + blk : T;
      for (int f = 0; f < d; ++f) {
        double sum = 0.0;
        for (int j = lo; j < hi; ++j) sum += kh[(size_t)j * d + f];
        mu[f] = sum / (hi - lo);
      }
      for (int i = lo; i < hi; ++i) a[T + i] = -or_cos(kh + (size_t)i * d, mu, d);
    }
    /* current anchor: causal moving mean */
    for (int i = 0; i < T; ++i) {
      const int lo = i - window + 1 > 0 ? i - window + 1 : 0;
      for (int f = 0; f < d; ++f) {
        double sum = 0.0;
        for (int j = lo; j <= i; ++j) sum += kh[(size_t)j * d + f];
        mu[f] = sum / (i - lo + 1);
      }
      a[2 * T + i] = -or_cos(kh + (size_t)i * d, mu, d);
    }
    /* discriminative power per scale and the softmax weights */
    double D[3], w[3];
    for (int k = 0; k < 3; ++k) {
      memcpy(srt, a + (size_t)k * T, sizeof(double) * (size_t)T);
      qsort(srt, (size_t)T, sizeof(double), or_cmp_double);
      double top = 0.0, bot = 0.0;
      for (int m = 0; m < n_disc; ++m) {
        bot += srt[m];
        top += srt[T - 1 - m];
      }
      D[k] = (top - bot) / n_disc;
    }
    double zmax = D[0] + log_prior[0];
    for (int k = 1; k < 3; ++k)
      if (D[k] + log_prior[k] > zmax) zmax = D[k] + log_prior[k];
    double zsum = 0.0;
    for (int k = 0; k < 3; ++k) {
      w[k] = exp(D[k] + log_prior[k] - zmax);
      zsum += w[k];
    }
    for (int k = 0; k < 3; ++k) w[k] /= zsum;
    /* blend, surprise, routing */
    for (int i = 0; i < T; ++i) {
      const double as = a[i], ae = a[T + i], ac = a[2 * T + i];
      const double blend = w[0] * as + w[1] * ae + w[2] * ac;
      const double mean = (as + ae + ac) / 3.0;
      const double sig = sqrt(((as - mean) * (as - mean) + (ae - mean) * (ae - mean) +
                               (ac - mean) * (ac - mean)) / 3.0);
      double win = as > ae ? as : ae;
      if (ac > win) win = ac;
      score_out[u * T + i] = sig > thresh ? win : blend;
      if (sigma_out) sigma_out[u * T + i] = sig;
    }
    if (a_out) memcpy(a_out + (size_t)u * 3 * T, a, sizeof(double) * 3 * (size_t)T);
    if (w_out)
      for (int k = 0; k < 3; ++k) w_out[u * 3 + k] = w[k];
    free(kh); free(a); free(srt); free(mu);
  }
  return bad ? -1 : 0;
}

/* ---------------------------------------------------------------------------
 * Step 5: one H2O decode step over a preallocated slot cache
 * ([H2O] 贪心驱逐算法, 问题形式化, FlexGen 改造).
 *
 * Per unit (b, h): the attended set C is the filled slots 0..len-1 plus the new
 * token (position new_pos), except with flag ALG1, where the new query attends
 * only to the cached tokens, as in Algorithm 1.  For each query head g of the
 * group: l_j = scale <q_g, k_j> over C, P = softmax over C (renormalised over the
 * kept keys only), o_g = sum_j P_j v_j.  Every cached accumulator gains the sum
 * over g of its P; the new token starts with its own sum (0 under ALG1).
 *   len < cap : the new token is appended in slot len; evicted = -1.
 *   len == cap: the victim is the argmin of (accumulator, position) over the
 *               slots with position <= new_pos - recent, plus the new token
 *               itself when recent == 0; the victim's slot is overwritten by the
 *               new token (K, V, position, accumulator) and evicted = its
 *               position; if the victim is the new token, nothing is written
 *               and evicted = new_pos.  At most one eviction per head per step.
 * With S sinks, slots holding positions below S are never victims either
 * ([KVblog] §4.1-4.2).
 * The accumulators are stored as float32 (their state type) and the argmin is
 * taken on the stored float32 values.
 * q [B][Hq][d]; k_new, v_new [B][Hkv][d]; K_cache, V_cache [B][Hkv][cap][d];
 * pos, acc [B][Hkv][cap]; len, evicted [B][Hkv]; o [B][Hq][d] (double).
 * ------------------------------------------------------------------------- */
int oracle_decode_step_ex(const void *q, const void *k_new, const void *v_new, void *K_cache,
                          void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq,
                          int Hkv, int cap, int d, int recent, int sink, int new_pos, double scale,
                          int flags, int dtype, double *o_out, int32_t *evicted) {
  const int alg1 = (flags & OR_FLAG_ALG1) != 0;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || cap <= 0 || d <= 0 || recent < 0 ||
      sink < 0 || recent >= cap || (alg1 && recent != 0))
    return -1;
  const int G = Hq / Hkv;
  const size_t eb = or_elem_bytes(dtype), row = (size_t)d * eb;
  const long long units = (long long)B * Hkv;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (long long u = 0; u < units; ++u) {
    const int b = (int)(u / Hkv), h = (int)(u % Hkv);
    const int n = len[u];
    if (n < 0 || n > cap) {
      bad = 1;
      continue;
    }
    const int with_self = !alg1;
    const int nc = n + with_self; /* attended set size */
    double *l = (double *)malloc(sizeof(double) * (size_t)(nc > 0 ? nc : 1));
    double *P = (double *)calloc((size_t)(nc > 0 ? nc : 1), sizeof(double));
    if (!l || !P) {
      free(l);
      free(P);
      bad = 1;
      continue;
    }
    const size_t kbase = ((size_t)u * cap) * (size_t)d;
    const size_t nbase = (size_t)u * (size_t)d;
    for (int g = 0; g < G; ++g) {
      const size_t qoff = ((size_t)b * Hq + (size_t)h * G + g) * (size_t)d;
      double *o = o_out + qoff;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      if (nc == 0) continue;
      double m = -INFINITY;
      for (int j = 0; j < nc; ++j) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c) {
          const double kv = (j < n) ? or_load(K_cache, kbase + (size_t)j * d + c, dtype)
                                    : or_load(k_new, nbase + c, dtype);
          dot += or_load(q, qoff + c, dtype) * kv;
        }
        l[j] = scale * dot;
        if (l[j] > m) m = l[j];
      }
      double Z = 0.0;
      for (int j = 0; j < nc; ++j) Z += exp(l[j] - m);
      for (int j = 0; j < nc; ++j) {
        const double p = exp(l[j] - m) / Z;
        P[j] += p;
        for (int c = 0; c < d; ++c) {
          const double vv = (j < n) ? or_load(V_cache, kbase + (size_t)j * d + c, dtype)
                                    : or_load(v_new, nbase + c, dtype);
          o[c] += p * vv;
        }
      }
    }
    float *a = acc + u * (long long)cap;
    int32_t *ps = pos + u * (long long)cap;
    for (int j = 0; j < n; ++j) a[j] = (float)((double)a[j] + P[j]);
    const float acc_new = with_self ? (float)P[n] : 0.0f;
    char *Kc = (char *)K_cache + (size_t)u * cap * row;
    char *Vc = (char *)V_cache + (size_t)u * cap * row;
    const char *kn = (const char *)k_new + (size_t)u * row;
    const char *vn = (const char *)v_new + (size_t)u * row;
    if (n < cap) {
      memcpy(Kc + (size_t)n * row, kn, row);
      memcpy(Vc + (size_t)n * row, vn, row);
      ps[n] = new_pos;
      a[n] = acc_new;
      len[u] = n + 1;
      evicted[u] = -1;
    } else {
      /* candidates: slots outside the protected recent window, and the new token
       * when no window protects it */
      int victim = -2; /* -2: none yet, -1: the new token */
      float best_acc = 0.0f;
      int best_pos = 0;
      for (int j = 0; j < n; ++j) {
        if ((long long)ps[j] > (long long)new_pos - recent) continue;
        if (ps[j] < sink) continue; /* a protected sink */
        if (victim == -2 || a[j] < best_acc || (a[j] == best_acc && ps[j] < best_pos)) {
          victim = j;
          best_acc = a[j];
          best_pos = ps[j];
        }
      }
      if (recent == 0) {
        if (victim == -2 || acc_new < best_acc || (acc_new == best_acc && new_pos < best_pos))
          victim = -1;
      }
      if (victim == -2) {
        bad = 1;
      } else if (victim == -1) {
        evicted[u] = new_pos;
      } else {
        evicted[u] = ps[victim];
        memcpy(Kc + (size_t)victim * row, kn, row);
        memcpy(Vc + (size_t)victim * row, vn, row);
        ps[victim] = new_pos;
        a[victim] = acc_new;
      }
    }
    free(l);
    free(P);
  }
  return bad ? -1 : 0;
}

int oracle_decode_step(const void *q, const void *k_new, const void *v_new, void *K_cache,
                       void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq,
                       int Hkv, int cap, int d, int recent, int new_pos, double scale,
                       int flags, int dtype, double *o_out, int32_t *evicted) {
  return oracle_decode_step_ex(q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq, Hkv, cap, d,
                               recent, 0, new_pos, scale, flags, dtype, o_out, evicted);
}
