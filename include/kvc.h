/*
 * kvc.h -- C ABI of libkvc.so, GB300 (sm_103a) KV-cache token eviction.
 *
 * The eviction path has five operations; each is one call here:
 *   kv_score_obs     observation-window attention mass per cached token
 *   hubkv_refine     HubKV score refinement before Top-K
 *   kv_select_topk   budgeted per-head Top-K with a protected recent window
 *   kv_compact       gather-compaction of the kept K/V rows into a slot cache
 *   h2o_decode_step  one decode step: attention, score accumulation, <= 1 eviction
 * and, beyond those five, NestedKV's key-only scorer (kv_score_nested), a
 * layer-level budget shared by the heads of a layer (kv_select_budget,
 * kv_compact_ragged) and the _ex variants (sinks, HubKV comparison variants).
 *
 * Sources (page title, section):
 *   [H2O]    "H2O 完全拆解：抓住 KV Cache 里的「重击者」，20% 预算无损生成（NeurIPS 2023）"
 *   [HubKV]  "HubKV walkthrough"
 *   [KVblog] the KV-cache survey blog (famous-torrone-8bc255.netlify.app/posts/kv_cache)
 *   [NestedKV] "Technische Samenvatting: NestedKV" (gist.science summary)
 *
 * Conventions shared by every call
 *   - Every pointer argument is DEVICE memory owned by the caller (allocate it
 *     with cudaMalloc or a framework allocator), 16-byte aligned; the gather
 *     sources of the two compactions may also be pinned host memory.  The library
 *     never allocates, frees or synchronises; it only enqueues kernels on
 *     `stream` (a cudaStream_t passed as void*, NULL = legacy default stream).
 *   - Tensors are dense, row-major, the head dimension fastest and the head
 *     index outside the token index: K is [B][Hkv][T][d], so one head's keys
 *     are one contiguous T x d block.  Layers are independent: a caller with L
 *     layers folds them into B.
 *   - `dtype` is KV_BF16 (bf16 storage, fp32 arithmetic) or KV_F32; it applies
 *     to Q, K, V, q, k_new, v_new and the caches.  Scores, accumulators and
 *     attention outputs are always float32.  d (head dimension) is 64 or 128.
 *   - Inputs must be finite; the kernels do not check (a check would cost a
 *     full extra pass over K).
 *   - Return value: KV_OK when the work was enqueued.  Argument errors
 *     (KV_ERR_INVALID_ARG, KV_ERR_UNSUPPORTED, KV_ERR_WORKSPACE) are returned
 *     before anything is launched and leave every output untouched.  A launch
 *     failure returns KV_ERR_CUDA.  Errors raised while kernels run (for example
 *     a bounded device-side wait that gave up) are written to `dev_status`
 *     where the call has one, and are visible after the caller synchronises.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVC_API __attribute__((visibility("default")))
#else
#define KVC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KV_OK = 0,
  KV_ERR_INVALID_ARG = -1, /* a size, pointer, alignment or flag is out of range */
  KV_ERR_UNSUPPORTED = -2, /* valid, but not a shape this build handles (e.g. d = 96) */
  KV_ERR_CUDA = -3,        /* the CUDA runtime refused the launch */
  KV_ERR_TIMEOUT = -4,     /* (device status) a bounded device-side wait gave up */
  KV_ERR_WORKSPACE = -5    /* workspace missing or smaller than kv_workspace_size() */
} kv_status;

typedef enum { KV_BF16 = 0, KV_F32 = 1 } kv_dtype;

/* h2o_decode_step flags */
enum {
  /* Algorithm 1 of [H2O] 贪心驱逐算法 exactly: the new query attends only to the
   * cached tokens (not to itself), the new token enters with accumulated score
   * 0 and competes for eviction at once.  Requires recent == 0. */
  KV_H2O_ALG1 = 1
};

/* hubkv_refine_ex flags: the variants [HubKV] 尝试路线：效果一般的可能原因 reports
 * as weaker than the final method, for comparison runs */
enum {
  /* average-pool smoothing ("CommunitySmooth") instead of steps 1-2: q_i = the
   * mean of s over the same window (cut at the ends) */
  KV_HUB_AVGPOOL = 1,
  /* fixed head weight instead of step 3: beta_h = 1 */
  KV_HUB_FIXED_HEAD = 2
};

/* operation codes for kv_workspace_size */
enum {
  KV_OP_SCORE_OBS = 1,
  KV_OP_HUBKV_REFINE = 2,
  KV_OP_SELECT_TOPK = 3,
  KV_OP_DECODE = 4,
  KV_OP_SCORE_NESTED = 5,
  KV_OP_HUBKV_SELECT = 6
};

typedef void *kv_stream_t;

/*
 * kv_score_obs -- per-head importance score of every prompt token.
 *
 * [H2O] 观察二 defines a token's score as the attention probability it has
 * accumulated; [KVblog] §4.3 (SnapKV) takes it from the prefill attention of an
 * observation window; [KVblog] §1.1 gives softmax(q.k / sqrt(d_head)).  For unit
 * (b, h) and each of its G = Hq/Hkv query heads g = h*G .. h*G+G-1 and window row
 * w (prompt position p = T - W + w):
 *     P_{g,w}(j) = softmax_j( scale * <Q_obs[b][g][w], K[b][h][j]> ),  j = 0..p
 *     s[b][h][j] = sum over g, w with p >= j of P_{g,w}(j)
 * Keys after a row's position get nothing from it (causal).  Hence
 * sum_j s[b][h][j] = G * W.
 *
 *   Q_obs      [B][Hq][W][d]   the last W prompt queries of every query head
 *   K          [B][Hkv][T][d]
 *   scale      logit scale, normally 1/sqrt(d)
 *   s_out      [B][Hkv][T] float32 (written in full)
 *   workspace  >= kv_workspace_size(KV_OP_SCORE_OBS, ...) bytes of device memory;
 *              its first words are cleared by an asynchronous memset on `stream`
 *              at the start of every call, the rest is written before it is read
 *   dev_status device int, may be NULL; set to KV_ERR_TIMEOUT if a bounded
 *              device-side wait gave up (s_out is then not valid); never cleared
 * Preconditions: 1 <= W <= T, Hq % Hkv == 0, d in {64, 128}.
 * bf16 inputs run on the tensor cores (tcgen05, TMA), the G*W query rows of a
 * unit in blocks of up to 256 (so W = T, every prompt query observed, works
 * too); fp32 inputs on the CUDA cores; both give the same quantity.  Repeated
 * calls on the same inputs give identical bits (fixed-order sums).
 */
KVC_API int kv_score_obs(const void *Q_obs, const void *K, int B, int Hq, int Hkv, int T, int d,
                 int W, float scale, int dtype, float *s_out, void *workspace,
                 size_t workspace_bytes, int *dev_status, kv_stream_t stream);

/*
 * hubkv_refine -- HubKV refinement of base scores before Top-K
 * ([HubKV] Method: 最终算法：四步修正原始分数).
 *   1. local hubs:  M_i = max_{|j-i| <= pool_width/2} s_j (window cut at the
 *                   ends); i is a hub iff s_i == M_i;
 *   2. SMD discount: q_i = s_i for a hub, gamma * s_i otherwise;
 *   3. head weight: sel_h = 1 - H(s_h / sum s_h) / ln T (normalised entropy,
 *                   0 ln 0 = 0; T == 1 or an all-zero head gives 0);
 *                   beta_h = clip(sel_h / mean_{h' in batch row} sel_h', beta_lo,
 *                   beta_hi), 1 when that mean is 0;
 *   4. ratio gate:  z_i = s_i + r^2 (beta_h q_i - s_i).
 * The head mean in step 3 runs over the H heads of one batch row b.
 *
 *   s          [B][H][T] float32 base scores (e.g. from kv_score_obs)
 *   z_out      [B][H][T] float32
 *   beta_out   [B][H] float32, may be NULL
 * Preconditions: pool_width odd, beta_lo <= beta_hi.
 */
KVC_API int hubkv_refine(const float *s, int B, int H, int T, int pool_width, float gamma, float r,
                 float beta_lo, float beta_hi, float *z_out, float *beta_out, void *workspace,
                 size_t workspace_bytes, kv_stream_t stream);

/*
 * hubkv_refine_ex -- hubkv_refine with `flags` (0 or KV_HUB_AVGPOOL |
 * KV_HUB_FIXED_HEAD) selecting the variants [HubKV] 尝试路线 compares against;
 * hubkv_refine is hubkv_refine_ex with flags = 0.  Other flag bits are rejected
 * with KV_ERR_INVALID_ARG.  Same arguments and workspace otherwise.
 */
KVC_API int hubkv_refine_ex(const float *s, int B, int H, int T, int pool_width, float gamma,
                    float r, float beta_lo, float beta_hi, int flags, float *z_out,
                    float *beta_out, void *workspace, size_t workspace_bytes, kv_stream_t stream);

/*
 * kv_select_topk -- budgeted per-head Top-K with a protected recent window.
 * [H2O] 双缓冲: the last `recent` positions [T-recent, T) are always kept; the
 * other k - recent slots go to the best of [0, T-recent) in the order
 * (z descending, position ascending).  Each head selects on its own
 * ([H2O] 为什么要按头独立驱逐).  idx_out lists the k kept positions of each
 * head in ascending order.  The selection is exact: the same z gives the same
 * idx bit for bit.
 *
 *   z          [B][H][T] float32 (finite; -0.0 is treated as +0.0)
 *   idx_out    [B][H][k] int32
 * Preconditions: 0 <= recent < k <= T.
 */
KVC_API int kv_select_topk(const float *z, int B, int H, int T, int k, int recent, int32_t *idx_out,
                   void *workspace, size_t workspace_bytes, kv_stream_t stream);

/*
 * kv_select_topk_ex -- kv_select_topk that also protects `sink` attention-sink
 * positions ([KVblog] §4.1-4.2: the first few tokens are kept, as StreamingLLM
 * keeps them with the recent window): [0, sink) and [T-recent, T) are always
 * kept and the k - recent - sink heavy slots go to the best of
 * [sink, T-recent) in the order (z descending, position ascending).
 * kv_select_topk is kv_select_topk_ex with sink = 0.
 * Preconditions: sink >= 0, 0 <= recent, sink + recent < k <= T.
 */
KVC_API int kv_select_topk_ex(const float *z, int B, int H, int T, int k, int recent, int sink,
                      int32_t *idx_out, void *workspace, size_t workspace_bytes,
                      kv_stream_t stream);

/*
 * hubkv_select_topk -- hubkv_refine_ex followed by kv_select_topk_ex, in one
 * call ([HubKV] Method: 最终算法 steps 1-4, then [H2O] 双缓冲 / 为什么要按头独立
 * 驱逐): the kept positions are exactly those kv_select_topk_ex returns on the z
 * that hubkv_refine_ex writes, and z_out / beta_out (when given) are bit for bit
 * what hubkv_refine_ex writes.  When the heads fit on chip (T - recent - sink <=
 * 393216) the selection kernel forms each candidate's z from s itself while
 * loading, so z never goes through device memory unless the caller asks for it.
 *
 *   s          [B][H][T] float32 base scores
 *   idx_out    [B][H][k] int32, kept positions ascending
 *   z_out      [B][H][T] float32, may be NULL
 *   beta_out   [B][H] float32, may be NULL
 *   workspace  >= kv_workspace_size(KV_OP_HUBKV_SELECT, B, H, H, T, 0, recent + sink, k)
 * Preconditions: those of hubkv_refine_ex and kv_select_topk_ex.
 */
KVC_API int hubkv_select_topk(const float *s, int B, int H, int T, int pool_width, float gamma,
                              float r, float beta_lo, float beta_hi, int flags, int k, int recent,
                              int sink, int32_t *idx_out, float *z_out, float *beta_out,
                              void *workspace, size_t workspace_bytes, kv_stream_t stream);

/*
 * kv_compact -- "real drop" gather-compaction ([H2O] 两套代码) into a
 * preallocated slot cache ([H2O] FlexGen 改造).  For every head and m < k:
 *     K_out[m] = K[idx[m]],  V_out[m] = V[idx[m]],  pos_out[m] = idx[m],
 *     acc_out[m] = s[idx[m]] (the attention mass received so far),
 * and len_out = k.  Slots k..cap-1 are not touched.  The copy is bit-exact.
 *
 *   K, V       [B][H][T][d]; device memory, or pinned host memory (allocated with
 *              cudaHostAlloc / cudaMallocHost, addressed through unified virtual
 *              addressing): the kernel then reads only the kept rows over the host
 *              link, so V of a host-resident prompt never has to move in full
 *   s          [B][H][T] float32, may be NULL (then acc_out is not written)
 *   idx        [B][H][k] int32, each in [0, T) (a slot whose index is out of
 *              range is left untouched)
 *   K_out, V_out [B][H][cap][d];  pos_out, acc_out [B][H][cap];  len_out [B][H]
 * Preconditions: k <= T, k <= cap; acc_out may be NULL.
 */
KVC_API int kv_compact(const void *K, const void *V, const float *s, const int32_t *idx, int B, int H,
               int T, int k, int d, int dtype, void *K_out, void *V_out, int cap,
               int32_t *pos_out, float *acc_out, int32_t *len_out, kv_stream_t stream);

/*
 * kv_score_nested -- NestedKV key-only importance scores ([NestedKV]
 * 1. Continuum Geheugentoestand, 2. Buitenste Leraar).  No queries: for unit
 * (b, h) over its T keys, with kh_i = k_i / |k_i| (0 for a zero key),
 *   stable    mu_s    = mean of kh over all T keys;
 *   episodic  mu_e(i) = mean of kh over i's block, blocks of ceil(T / n_blocks)
 *                       consecutive keys (the pages: b ~ N/32, so n_blocks = 32);
 *   current   mu_c(i) = mean of kh over [max(0, i - window + 1), i] (causal
 *                       moving mean, i included; the pages: window = 64);
 *   a_k(i)  = -cos(k_i, mu_k(i)), 0 when a norm is 0 (high = anomalous = keep);
 *   D_k     = mean of the n_disc largest a_k(i) - mean of the n_disc smallest
 *             (each scale's discriminative power in this head);
 *   w       = softmax over k of D_k + log_prior_k (the fixed log-prior);
 *   sigma(i)= population standard deviation of (a_s, a_e, a_c)(i) (surprise);
 *   score(i)= max_k a_k(i) if sigma(i) > surprise_thresh, else sum_k w_k a_k(i).
 * The scores rank tokens for kv_select_topk / kv_select_budget.
 *
 *   K          [B][H][T][d] (dtype as everywhere; fp32 arithmetic)
 *   score_out  [B][H][T] float32
 *   w_out      [B][H][3] float32 (w_s, w_e, w_c), may be NULL
 *   a_out      [B][H][3][T] float32 (a_s, a_e, a_c), may be NULL; when given it
 *              also serves as their scratch, so the workspace can be smaller
 *   workspace  >= kv_workspace_size(KV_OP_SCORE_NESTED, B, 0, H, T, d, n_blocks, 0)
 *              bytes (that size assumes a_out == NULL)
 * Preconditions: 1 <= window <= 4096, 1 <= n_blocks <= 65536, 1 <= n_disc <= T,
 * finite log priors, surprise_thresh not NaN, d in {64, 128}.
 * Four launches: two key scans (the stable anchor needs every key before any
 * score), one selection per (unit, scale), one elementwise pass.
 */
KVC_API int kv_score_nested(const void *K, int B, int H, int T, int d, int dtype, int window,
                            int n_blocks, int n_disc, float log_prior_s, float log_prior_e,
                            float log_prior_c, float surprise_thresh, float *score_out,
                            float *w_out, float *a_out, void *workspace, size_t workspace_bytes,
                            kv_stream_t stream);

/*
 * kv_select_budget -- layer-level competitive budget: the heads of one layer
 * share one budget ([NestedKV] 3. Hoofd-gewijze Geheugentoewijzing: the
 * (token, head) pairs with the highest scores across the layer win, every head
 * keeping a minimum; [KVblog] §4.4 PyramidKV: budgets per layer, not per head).
 * Batch row b is one layer (fold batch x layers into B); its H heads keep
 * `budget` positions in all:
 *   1. every head keeps its sinks [0, sink) and its recent window [T-recent, T);
 *   2. floor: every head keeps its floor_k - sink - recent best positions of
 *      [sink, T-recent) in the order (z descending, position ascending), so each
 *      head keeps at least floor_k;
 *   3. competition: the budget - H*floor_k slots left go to the best of the
 *      row's (head, position) pairs with position in [sink, T-recent) not kept
 *      yet, in the order (z descending, head ascending, position ascending).
 * Steps 2-3 keep the largest score sum among all sets that keep the protected
 * positions, at least floor_k per head and budget in all.  The result is exact:
 * the same z gives the same output bit for bit.
 *
 *   z          [B][H][T] float32 (finite; -0.0 is treated as +0.0), 16-byte aligned
 *   idx_out    [B][budget] int32: head h's kept positions, ascending, at
 *              idx_out[b][off_out[b][h] .. off_out[b][h+1]-1]
 *   off_out    [B][H+1] int32: off_out[b][0] = 0, off_out[b][H] = budget
 * Preconditions: 0 <= sink, 0 <= recent, max(1, sink + recent) <= floor_k <= T,
 * H*floor_k <= budget <= H*T.  H <= 256 and H*T < 2^31 (else KV_ERR_UNSUPPORTED).
 * No workspace.  Runs one thread-block cluster of min(H, 8) CTAs per row.
 */
KVC_API int kv_select_budget(const float *z, int B, int H, int T, int budget, int floor_k,
                             int recent, int sink, int32_t *idx_out, int32_t *off_out,
                             kv_stream_t stream);

/*
 * kv_compact_ragged -- kv_compact for the per-head counts of kv_select_budget.
 * Head h of row b keeps n = off[b][h+1] - off[b][h] rows: for m < n,
 *     K_out[m] = K[idx[b][off[b][h] + m]], V_out[m] = V[...], pos_out[m] = that
 *     index, acc_out[m] = s[that index],
 * and len_out = n; slots n..cap-1 are not touched.  The copy is bit-exact.
 *
 *   K, V       [B][H][T][d], device or pinned host memory (as for kv_compact);
 *              s [B][H][T] float32, may be NULL (acc_out not written)
 *   idx        [B][budget] int32 (may be NULL when budget == 0);  off [B][H+1] int32
 *              (CSR, as kv_select_budget writes)
 *   K_out, V_out [B][H][cap][d];  pos_out, acc_out [B][H][cap];  len_out [B][H]
 *   dev_status device int, may be NULL; set to KV_ERR_INVALID_ARG when a row's
 *              offsets are not non-decreasing within [0, budget] (that row is left
 *              untouched) or a head keeps more than cap rows (that head is left
 *              untouched); never cleared.  An index outside [0, T) leaves its slot
 *              untouched.
 * Preconditions: d in {64, 128}, H <= 256; acc_out may be NULL.
 */
KVC_API int kv_compact_ragged(const void *K, const void *V, const float *s, const int32_t *idx,
                              const int32_t *off, int B, int H, int T, int budget, int d,
                              int dtype, void *K_out, void *V_out, int cap, int32_t *pos_out,
                              float *acc_out, int32_t *len_out, int *dev_status,
                              kv_stream_t stream);

/*
 * h2o_decode_step -- one decode step of the H2O eviction policy over a slot
 * cache ([H2O] 问题形式化, 贪心驱逐算法, 双缓冲, FlexGen 改造).
 * Per unit (b, h): the attended set C is the filled slots 0..len-1 plus the new
 * token (unless KV_H2O_ALG1).  For each query head g of the group:
 *     P_g = softmax over C of scale * <q_g, k_j>  (renormalised over kept keys),
 *     o_out[b][g] = sum_j P_g(j) v_j.
 * Each cached accumulator gains sum_g P_g(j); the new token starts with its own
 * sum (0 under KV_H2O_ALG1).  Then:
 *   len < cap : the new token goes to slot len, len += 1, evicted_pos = -1;
 *   len == cap: the victim is the smallest (acc, pos) among the slots with
 *               pos <= new_pos - recent (the new token itself also competes
 *               when recent == 0); its slot is overwritten in place by the new
 *               token (K, V, pos, acc) and evicted_pos = the victim's position;
 *               if the victim is the new token nothing is written and
 *               evicted_pos = new_pos.
 * At most one eviction per KV head per step; |cache| stays cap once full.
 *
 *   q          [B][Hq][d];  k_new, v_new [B][Hkv][d]
 *   K_cache, V_cache [B][Hkv][cap][d]   updated in place
 *   pos [B][Hkv][cap] int32, acc [B][Hkv][cap] float32, len [B][Hkv] int32 (in place)
 *   o_out [B][Hq][d] float32;  evicted_pos [B][Hkv] int32
 *   workspace  >= kv_workspace_size(KV_OP_DECODE, B, Hq, Hkv, cap, d, 0, 0) bytes
 *   dev_status  device int, may be NULL; set to a kv_status if a device-side
 *               error occurs (e.g. a len outside [0, cap]: that unit is then left
 *               untouched), never cleared by the library
 * Preconditions: 0 <= recent < cap, KV_H2O_ALG1 => recent == 0, new_pos larger
 * than every cached position, 0 <= len <= cap.
 * With B >= 2 the batch rows run in two halves, [0, B/2) on `stream` and the
 * rest on a library-owned stream of the current device (created on first use),
 * forked from and joined back into `stream` with events: the call stays
 * asynchronous and ordered on `stream` (and can be captured into a graph), and
 * one half's finalize work overlaps the other half's cache pass.  The
 * workspace holds both halves' scratch (kv_workspace_size accounts for it).
 */
KVC_API int h2o_decode_step(const void *q, const void *k_new, const void *v_new, void *K_cache,
                    void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq,
                    int Hkv, int cap, int d, int recent, int32_t new_pos, float scale,
                    int flags, int dtype, float *o_out, int32_t *evicted_pos, void *workspace,
                    size_t workspace_bytes, int *dev_status, kv_stream_t stream);

/*
 * h2o_decode_step_ex -- h2o_decode_step that also protects attention sinks
 * ([KVblog] §4.1-4.2): a slot holding a position below `sink` is never a victim
 * (it keeps accumulating like any other slot).  h2o_decode_step is
 * h2o_decode_step_ex with sink = 0.  Same arguments and workspace otherwise;
 * sink < 0 is rejected with KV_ERR_INVALID_ARG.
 */
KVC_API int h2o_decode_step_ex(const void *q, const void *k_new, const void *v_new, void *K_cache,
                       void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq,
                       int Hkv, int cap, int d, int recent, int sink, int32_t new_pos,
                       float scale, int flags, int dtype, float *o_out, int32_t *evicted_pos,
                       void *workspace, size_t workspace_bytes, int *dev_status,
                       kv_stream_t stream);

/*
 * h2o_decode_steps -- n_steps consecutive decode steps in one call: step t
 * (t = 0 .. n_steps-1) is h2o_decode_step_ex with q + t*B*Hq*d, k_new/v_new +
 * t*B*Hkv*d, new_pos = first_pos + t, o_out + t*B*Hq*d and evicted_pos +
 * t*B*Hkv.  The steps are enqueued back to back on `stream` (two launches each),
 * which removes a caller's per-step launch overhead when the queries are known
 * ahead.  The result is exactly that of the n_steps single calls.
 *
 *   q          [n_steps][B][Hq][d];  k_new, v_new [n_steps][B][Hkv][d]
 *   o_out      [n_steps][B][Hq][d] float32;  evicted_pos [n_steps][B][Hkv] int32
 *   everything else as for h2o_decode_step_ex (state updated in place)
 * Preconditions: n_steps >= 0, first_pos + n_steps - 1 fits int32, and those of
 * h2o_decode_step_ex.
 */
KVC_API int h2o_decode_steps(const void *q, const void *k_new, const void *v_new, int n_steps,
                             void *K_cache, void *V_cache, int32_t *pos, float *acc, int32_t *len,
                             int B, int Hq, int Hkv, int cap, int d, int recent, int sink,
                             int32_t first_pos, float scale, int flags, int dtype, float *o_out,
                             int32_t *evicted_pos, void *workspace, size_t workspace_bytes,
                             int *dev_status, kv_stream_t stream);

/*
 * kv_score_obs_noalloc -- kv_score_obs without a caller-provided workspace.
 * (No counterpart in the pages: this is a calling convention, not a step of
 * the method.)
 *
 * For callers that cannot allocate device memory: code embedded in a host
 * framework that hands it only its input and output buffers, and code that
 * must not call cudaMalloc because that call can synchronise the device and
 * stall other streams.  Computes exactly what kv_score_obs computes, with the
 * same arguments minus the workspace, using scratch space from a fixed array
 * of KV_SCORE_NOALLOC_SCRATCH_BYTES bytes inside the library's device image;
 * it allocates nothing.
 *   - Every GPU that loads the library holds that array until the process exits.
 *   - Shapes that need more scratch than that (kv_workspace_size(
 *     KV_OP_SCORE_OBS, ...) > KV_SCORE_NOALLOC_SCRATCH_BYTES) are rejected with
 *     KV_ERR_WORKSPACE before anything is launched.
 *   - All calls share the one array: calls that overlap on the GPU (different
 *     streams, or different host threads) race and corrupt each other's
 *     results, so serialise them.  The array keeps the last call's contents;
 *     each call clears the few words that must start at zero (the kernels'
 *     work-claim counters) with a memset on `stream` before its kernels run.
 *   - The first call on each device looks the array's device address up, with
 *     that device current; make that first call before any stream capture.
 *     The address is kept for the life of the process: it is not valid after
 *     cudaDeviceReset (or any other teardown of the device's primary context),
 *     so do not call this entry point again after one.
 */
#define KV_SCORE_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
KVC_API int kv_score_obs_noalloc(const void *Q_obs, const void *K, int B, int Hq, int Hkv, int T,
                                 int d, int W, float scale, int dtype, float *s_out,
                                 int *dev_status, kv_stream_t stream);

/* Device workspace (bytes) that `op` needs for these sizes; 0 if none.
 * Arguments that an op does not use are ignored; for KV_OP_HUBKV_REFINE pass the
 * refine call's head count H as Hkv; for KV_OP_DECODE pass the slot capacity as T;
 * for KV_OP_SCORE_NESTED pass H as Hkv and n_blocks as W.
 * Returns 0 for invalid sizes. */
KVC_API size_t kv_workspace_size(int op, int B, int Hq, int Hkv, int T, int d, int W, int k);

/* Static description of a kv_status value. */
KVC_API const char *kv_status_string(int status);

/* Library version (major * 10000 + minor * 100 + patch). */
KVC_API int kv_version(void);

/* Text of the CUDA error behind the calling thread's last KV_ERR_CUDA (the
 * failing step, the CUDA error string and name), "" before any; the pointer
 * stays valid in that thread until its next failing call.  Diagnostic only. */
KVC_API const char *kv_last_error_detail(void);

/* Number of kernels this library has launched in this process (all devices,
 * all threads); a diagnostic for counting launches around a timed region. */
KVC_API unsigned long long kv_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
