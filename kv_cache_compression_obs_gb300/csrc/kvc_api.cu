// kvc_api.cu -- the extern "C" entry points of libkvc.so: argument checks, then
// one launcher per operation.  Every check runs on the host before anything is
// enqueued, so a rejected call touches neither the GPU nor any output.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>
#include <mutex>
#include <unordered_map>

#include "kvc_internal.cuh"

namespace kvc {

static std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

namespace {
thread_local char g_detail[256] = "";
}
int cuda_failure(cudaError_t e, const char *where) {
  snprintf(g_detail, sizeof g_detail, "%s: %s (%s)", where, cudaGetErrorString(e), cudaGetErrorName(e));
  return KV_ERR_CUDA;
}
const char *last_detail() { return g_detail; }

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kNumSmsHint;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return kNumSmsHint;
  return n;
}

// Raise a kernel's dynamic shared-memory limit once per (device, kernel) when its
// static plus dynamic shared memory passes the 48 KB default.
int ensure_smem(const void *func, size_t bytes) {
  struct Entry {
    size_t static_bytes = 0;  // the kernel's static shared memory
    size_t granted = 0;       // dynamic bytes it has been opted into
  };
  static std::mutex mu;
  static std::unordered_map<const void *, Entry> done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(mu);
  auto it = done[dev].find(func);
  if (it == done[dev].end()) {  // first launch of this kernel on this device
    cudaFuncAttributes fa = {};
    if (cudaFuncGetAttributes(&fa, func) != cudaSuccess) {
      cudaGetLastError();
      return 1;
    }
    Entry e;
    e.static_bytes = fa.sharedSizeBytes;
    e.granted = e.static_bytes <= 48 * 1024 ? 48 * 1024 - e.static_bytes : 0;
    it = done[dev].emplace(func, e).first;
  }
  Entry &e = it->second;
  if (bytes <= e.granted) return 0;
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if ((size_t)optin < bytes + e.static_bytes) return 1;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
      cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  e.granted = bytes;
  return 0;
}

// Argument checks of the scoring entry points (kv_score_obs and its no-alloc
// variant), in one place so both answer alike.  KV_OK with B == 0 means there is
// nothing to launch.
int check_score_args(const void *Q_obs, const void *K, int B, int Hq, int Hkv, int T, int d,
                     int W, float scale, int dtype, const float *s_out) {
  auto fits = [](long long a, long long b) { return a >= 0 && b >= 0 && (b == 0 || a <= (1LL << 62) / b); };
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || T <= 0 || W <= 0 || W > T ||
      !(dtype == KV_BF16 || dtype == KV_F32) || !(scale == scale))
    return KV_ERR_INVALID_ARG;
  if (!(d == 64 || d == 128)) return KV_ERR_UNSUPPORTED;
  if (!fits((long long)B * Hkv, (long long)T * d) || !fits((long long)B * Hq, (long long)W * d))
    return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  if (!Q_obs || !K || !s_out || !aligned16(Q_obs) || !aligned16(K) || !aligned16(s_out))
    return KV_ERR_INVALID_ARG;
  return KV_OK;
}

}  // namespace kvc

using namespace kvc;

namespace {

bool dtype_ok(int dt) { return dt == KV_BF16 || dt == KV_F32; }
bool dim_ok(int d) { return d == 64 || d == 128; }
// product of non-negative ints without overflow of 2^62
bool fits(long long a, long long b) { return a >= 0 && b >= 0 && (b == 0 || a <= (1LL << 62) / b); }


// A decode call's batch rows run in two halves: rows [0, B/2) on the caller's
// stream and [B/2, B) on a library-owned side stream (one per device, created on
// first use), forked from and joined back into the caller's stream with events.
// The halves are independent units; each half's latency-bound finalize launches
// run beside the other half's bandwidth-bound stream kernel.  Fewer than 2 rows,
// or a device whose side stream could not be created, run on the caller's
// stream alone.
int split_rows(int B) { return B >= 2 ? B / 2 : B; }

size_t align256h(size_t x) { return (x + 255) & ~(size_t)255; }

size_t decode_ws_split(int B, int Hkv, int G, int cap, int d) {
  const int Ba = split_rows(B);
  const size_t a = decode_workspace_bytes((long)Ba * Hkv, G, cap, d);
  if (Ba == B) return a;
  return align256h(a) + decode_workspace_bytes((long)(B - Ba) * Hkv, G, cap, d);
}

struct SideStream {
  std::mutex mu;
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool ready = false, failed = false;
};
SideStream g_side[64];

int decode_run(const void *q, const void *k_new, const void *v_new, int n_steps, void *K_cache,
               void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq, int Hkv,
               int cap, int d, int recent, int sink, int32_t first_pos, float scale, int flags,
               int dtype, float *o_out, int32_t *evicted_pos, void *workspace, int *dev_status,
               cudaStream_t stream) {
  const size_t eb = dtype == KV_F32 ? 4 : 2;
  const int G = Hq / Hkv;
  // step t of rows [r0, r1)
  auto step = [&](int t, int r0, int r1, void *ws, cudaStream_t st) {
    const size_t row_q = (size_t)Hq * d, row_kv = (size_t)Hkv * d, row_c = (size_t)Hkv * cap;
    const size_t qo = ((size_t)t * B + r0) * row_q, ko = ((size_t)t * B + r0) * row_kv;
    return launch_decode_step(
        static_cast<const char *>(q) + qo * eb, static_cast<const char *>(k_new) + ko * eb,
        static_cast<const char *>(v_new) + ko * eb,
        static_cast<char *>(K_cache) + (size_t)r0 * row_c * d * eb,
        static_cast<char *>(V_cache) + (size_t)r0 * row_c * d * eb, pos + (size_t)r0 * row_c,
        acc + (size_t)r0 * row_c, len + (size_t)r0 * Hkv, r1 - r0, Hq, Hkv, cap, d, recent, sink,
        first_pos + t, scale, flags, dtype, ws, o_out + qo,
        evicted_pos + ((size_t)t * B + r0) * Hkv, dev_status, st);
  };
  auto single = [&]() {
    for (int t = 0; t < n_steps; ++t) {
      const int rc = step(t, 0, B, workspace, stream);
      if (rc != KV_OK) return rc;
    }
    return (int)KV_OK;
  };
  const int Ba = split_rows(B);
  int dev = 0;
  if (Ba == B || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return single();
  SideStream &sd = g_side[dev];
  std::lock_guard<std::mutex> lock(sd.mu);
  if (!sd.ready && !sd.failed) {
    if (cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking) == cudaSuccess &&
        cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) == cudaSuccess &&
        cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) == cudaSuccess) {
      sd.ready = true;
    } else {
      cudaGetLastError();
      sd.failed = true;  // the whole batch then runs on the caller's stream
    }
  }
  if (!sd.ready) return single();
  void *ws_b = static_cast<char *>(workspace) +
               align256h(decode_workspace_bytes((long)Ba * Hkv, G, cap, d));
  cudaError_t e = cudaEventRecord(sd.fork, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(sd.s, sd.fork, 0);
  if (e != cudaSuccess) return cuda_failure(e, "decode: fork to the side stream");
  int rc = KV_OK;
  for (int t = 0; t < n_steps && rc == KV_OK; ++t) {  // interleaved, so both streams start at once
    rc = step(t, 0, Ba, workspace, stream);
    if (rc == KV_OK) rc = step(t, Ba, B, ws_b, sd.s);
  }
  e = cudaEventRecord(sd.join, sd.s);  // joined back even after a failed launch
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, sd.join, 0);
  if (e != cudaSuccess && rc == KV_OK) rc = cuda_failure(e, "decode: join from the side stream");
  return rc;
}

}  // namespace

extern "C" {


int kv_version(void) { return 100; }

unsigned long long kv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *kv_last_error_detail(void) { return kvc::last_detail(); }

const char *kv_status_string(int status) {
  switch (status) {
    case KV_OK: return "ok";
    case KV_ERR_INVALID_ARG: return "invalid argument";
    case KV_ERR_UNSUPPORTED: return "unsupported shape or option";
    case KV_ERR_CUDA: return "CUDA launch error";
    case KV_ERR_TIMEOUT: return "device-side wait timed out";
    case KV_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

size_t kv_workspace_size(int op, int B, int Hq, int Hkv, int T, int d, int W, int k) {
  (void)d;
  if (B < 0 || T <= 0) return 0;
  switch (op) {
    case KV_OP_SCORE_OBS:
      if (Hq <= 0 || Hkv <= 0 || Hq % Hkv || W <= 0 || W > T) return 0;
      return plan_score(B, Hq, Hkv, T, W).ws_bytes;
    case KV_OP_HUBKV_REFINE:
      if (Hkv <= 0) return 0;
      return plan_refine(B, Hkv, T).ws_bytes;  // the refine call's H is passed as Hkv
    case KV_OP_SELECT_TOPK:
      return 0;
    case KV_OP_HUBKV_SELECT: {  // the refine call's H is passed as Hkv, recent + sink as W
      if (Hkv <= 0 || W < 0 || k <= W || k > T) return 0;
      const size_t r = align256h(plan_refine(B, Hkv, T).ws_bytes);
      return r + (hubkv_select_needs_z(T, k, W, 0) ? (size_t)B * Hkv * T * sizeof(float) : 0);
    }
    case KV_OP_SCORE_NESTED:  // Hkv is the head count, W the number of episodic blocks
      if (Hkv <= 0 || W <= 0 || !(d == 64 || d == 128)) return 0;
      return nested_workspace_bytes((long)B * Hkv, T, d, W, true);
    case KV_OP_DECODE:  // T is the slot capacity
      if (Hq <= 0 || Hkv <= 0 || Hq % Hkv || !(d == 64 || d == 128)) return 0;
      return decode_ws_split(B, Hkv, Hq / Hkv, T, d);
    default:
      return 0;
  }
}

int kv_score_obs(const void *Q_obs, const void *K, int B, int Hq, int Hkv, int T, int d, int W,
                 float scale, int dtype, float *s_out, void *workspace, size_t workspace_bytes,
                 int *dev_status, kv_stream_t stream) {
  const int rc = kvc::check_score_args(Q_obs, K, B, Hq, Hkv, T, d, W, scale, dtype, s_out);
  if (rc != KV_OK || B == 0) return rc;
  const ScorePlan plan = plan_score(B, Hq, Hkv, T, W);
  if (!workspace || workspace_bytes < plan.ws_bytes || !aligned16(workspace)) return KV_ERR_WORKSPACE;
  return launch_score_obs(Q_obs, K, B, Hq, Hkv, T, d, W, scale, dtype, s_out, workspace, plan,
                          dev_status, static_cast<cudaStream_t>(stream));
}

int hubkv_refine_ex(const float *s, int B, int H, int T, int pool_width, float gamma, float r,
                    float beta_lo, float beta_hi, int flags, float *z_out, float *beta_out,
                    void *workspace, size_t workspace_bytes, kv_stream_t stream) {
  if (B < 0 || H <= 0 || T <= 0 || pool_width <= 0 || pool_width % 2 == 0 ||
      !(beta_lo <= beta_hi) || !(gamma == gamma) || !(r == r) ||
      (flags & ~(KV_HUB_AVGPOOL | KV_HUB_FIXED_HEAD)))
    return KV_ERR_INVALID_ARG;
  if (pool_width > 129) return KV_ERR_UNSUPPORTED;
  if (!fits((long long)B * H, T)) return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  if (!s || !z_out || !aligned16(s) || !aligned16(z_out)) return KV_ERR_INVALID_ARG;
  const RefinePlan plan = plan_refine(B, H, T);
  if (!workspace || workspace_bytes < plan.ws_bytes || !aligned16(workspace)) return KV_ERR_WORKSPACE;
  return launch_hubkv_refine(s, B, H, T, pool_width, gamma, r, beta_lo, beta_hi, flags, z_out,
                             beta_out, workspace, plan, static_cast<cudaStream_t>(stream));
}

int hubkv_refine(const float *s, int B, int H, int T, int pool_width, float gamma, float r,
                 float beta_lo, float beta_hi, float *z_out, float *beta_out, void *workspace,
                 size_t workspace_bytes, kv_stream_t stream) {
  return hubkv_refine_ex(s, B, H, T, pool_width, gamma, r, beta_lo, beta_hi, 0, z_out, beta_out,
                         workspace, workspace_bytes, stream);
}

int hubkv_select_topk(const float *s, int B, int H, int T, int pool_width, float gamma, float r,
                      float beta_lo, float beta_hi, int flags, int k, int recent, int sink,
                      int32_t *idx_out, float *z_out, float *beta_out, void *workspace,
                      size_t workspace_bytes, kv_stream_t stream) {
  if (B < 0 || H <= 0 || T <= 0 || pool_width <= 0 || pool_width % 2 == 0 ||
      !(beta_lo <= beta_hi) || !(gamma == gamma) || !(r == r) ||
      (flags & ~(KV_HUB_AVGPOOL | KV_HUB_FIXED_HEAD)) || recent < 0 || sink < 0 ||
      k <= recent + sink || k > T)
    return KV_ERR_INVALID_ARG;
  if (pool_width > 129) return KV_ERR_UNSUPPORTED;
  if (!fits((long long)B * H, T)) return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  if (!s || !idx_out || !aligned16(s) || !aligned16(idx_out) || (z_out && !aligned16(z_out)))
    return KV_ERR_INVALID_ARG;
  const RefinePlan plan = plan_refine(B, H, T);
  const size_t rbytes = align256h(plan.ws_bytes);
  const bool need_z = hubkv_select_needs_z(T, k, recent, sink);
  const size_t need = rbytes + (need_z ? (size_t)B * H * T * sizeof(float) : 0);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return KV_ERR_WORKSPACE;
  float *z_tmp = need_z ? reinterpret_cast<float *>(static_cast<char *>(workspace) + rbytes) : nullptr;
  return launch_hubkv_select(s, B, H, T, pool_width, gamma, r, beta_lo, beta_hi, flags, k, recent,
                             sink, idx_out, z_out, beta_out, workspace, plan, z_tmp,
                             static_cast<cudaStream_t>(stream));
}

int kv_select_topk_ex(const float *z, int B, int H, int T, int k, int recent, int sink,
                      int32_t *idx_out, void *workspace, size_t workspace_bytes, kv_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (B < 0 || H <= 0 || T <= 0 || recent < 0 || sink < 0 || k <= recent + sink || k > T)
    return KV_ERR_INVALID_ARG;
  if (!fits((long long)B * H, T)) return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  if (!z || !idx_out || !aligned16(z) || !aligned16(idx_out)) return KV_ERR_INVALID_ARG;
  return launch_select_topk(z, B, H, T, k, recent, sink, idx_out, static_cast<cudaStream_t>(stream));
}

int kv_select_topk(const float *z, int B, int H, int T, int k, int recent, int32_t *idx_out,
                   void *workspace, size_t workspace_bytes, kv_stream_t stream) {
  return kv_select_topk_ex(z, B, H, T, k, recent, 0, idx_out, workspace, workspace_bytes, stream);
}

int kv_compact(const void *K, const void *V, const float *s, const int32_t *idx, int B, int H,
               int T, int k, int d, int dtype, void *K_out, void *V_out, int cap,
               int32_t *pos_out, float *acc_out, int32_t *len_out, kv_stream_t stream) {
  if (B < 0 || H <= 0 || T <= 0 || k <= 0 || k > T || cap < k || !dtype_ok(dtype))
    return KV_ERR_INVALID_ARG;
  if (!dim_ok(d)) return KV_ERR_UNSUPPORTED;
  if (!fits((long long)B * H, (long long)T * d) || !fits((long long)B * H, (long long)cap * d))
    return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  if (!K || !V || !idx || !K_out || !V_out || !pos_out || !len_out) return KV_ERR_INVALID_ARG;
  if (!aligned16(K) || !aligned16(V) || !aligned16(K_out) || !aligned16(V_out) ||
      (s && !aligned16(s)) || (acc_out && !aligned16(acc_out)))
    return KV_ERR_INVALID_ARG;
  return launch_compact(K, V, acc_out ? s : nullptr, idx, B, H, T, k, d, dtype, K_out, V_out,
                        cap, pos_out, acc_out, len_out, static_cast<cudaStream_t>(stream));
}

int kv_select_budget(const float *z, int B, int H, int T, int budget, int floor_k, int recent,
                     int sink, int32_t *idx_out, int32_t *off_out, kv_stream_t stream) {
  if (B < 0 || H <= 0 || T <= 0 || recent < 0 || sink < 0 || floor_k < 1 ||
      floor_k < recent + sink || floor_k > T || (long long)budget < (long long)H * floor_k ||
      (long long)budget > (long long)H * T)
    return KV_ERR_INVALID_ARG;
  if (H > 256 || (long long)H * T > INT_MAX) return KV_ERR_UNSUPPORTED;
  if (!fits(B, budget)) return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  if (!z || !idx_out || !off_out || !aligned16(z) || ((uintptr_t)idx_out & 3u) ||
      ((uintptr_t)off_out & 3u))
    return KV_ERR_INVALID_ARG;
  return launch_select_budget(z, B, H, T, budget, floor_k, recent, sink, idx_out, off_out,
                              static_cast<cudaStream_t>(stream));
}

int kv_compact_ragged(const void *K, const void *V, const float *s, const int32_t *idx,
                      const int32_t *off, int B, int H, int T, int budget, int d, int dtype,
                      void *K_out, void *V_out, int cap, int32_t *pos_out, float *acc_out,
                      int32_t *len_out, int *dev_status, kv_stream_t stream) {
  if (B < 0 || H <= 0 || T <= 0 || budget < 0 || cap < 0 || !dtype_ok(dtype))
    return KV_ERR_INVALID_ARG;
  if (!dim_ok(d)) return KV_ERR_UNSUPPORTED;
  if (H > 256) return KV_ERR_UNSUPPORTED;
  if (!fits((long long)B * H, (long long)T * d) || !fits((long long)B * H, (long long)cap * d) ||
      !fits(B, budget))
    return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  if (!K || !V || (!idx && budget > 0) || !off || !K_out || !V_out || !pos_out || !len_out)
    return KV_ERR_INVALID_ARG;  // idx is not read when the budget is 0
  if (!aligned16(K) || !aligned16(V) || !aligned16(K_out) || !aligned16(V_out) ||
      (s && ((uintptr_t)s & 3u)) || (acc_out && ((uintptr_t)acc_out & 3u)))
    return KV_ERR_INVALID_ARG;
  return launch_compact_ragged(K, V, acc_out ? s : nullptr, idx, off, B, H, T, budget, d, dtype,
                               K_out, V_out, cap, pos_out, acc_out, len_out, dev_status,
                               static_cast<cudaStream_t>(stream));
}

int kv_score_nested(const void *K, int B, int H, int T, int d, int dtype, int window,
                    int n_blocks, int n_disc, float log_prior_s, float log_prior_e,
                    float log_prior_c, float surprise_thresh, float *score_out, float *w_out,
                    float *a_out, void *workspace, size_t workspace_bytes, kv_stream_t stream) {
  if (B < 0 || H <= 0 || T <= 0 || !dtype_ok(dtype) || window < 1 || n_blocks < 1 ||
      n_disc < 1 || n_disc > T || !(surprise_thresh == surprise_thresh) ||
      !std::isfinite(log_prior_s) || !std::isfinite(log_prior_e) || !std::isfinite(log_prior_c))
    return KV_ERR_INVALID_ARG;
  if (!dim_ok(d)) return KV_ERR_UNSUPPORTED;
  if (window > 4096 || n_blocks > 65536) return KV_ERR_UNSUPPORTED;
  if (!fits((long long)B * H, (long long)T * d) || !fits((long long)B * H, n_blocks) ||
      (long long)B * H * n_blocks > INT_MAX || (long long)B * H * 3 > INT_MAX)
    return KV_ERR_INVALID_ARG;
  if (B == 0) return KV_OK;
  if (!K || !score_out || !aligned16(K) || ((uintptr_t)score_out & 3u) ||
      (w_out && ((uintptr_t)w_out & 3u)) || (a_out && ((uintptr_t)a_out & 3u)))
    return KV_ERR_INVALID_ARG;
  const size_t need = nested_workspace_bytes((long)B * H, T, d, n_blocks, a_out == nullptr);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return KV_ERR_WORKSPACE;
  return launch_score_nested(K, B, H, T, d, dtype, window, n_blocks, n_disc, log_prior_s,
                             log_prior_e, log_prior_c, surprise_thresh, score_out, w_out, a_out,
                             workspace, static_cast<cudaStream_t>(stream));
}

int h2o_decode_step_ex(const void *q, const void *k_new, const void *v_new, void *K_cache,
                    void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq,
                    int Hkv, int cap, int d, int recent, int sink, int32_t new_pos, float scale,
                    int flags, int dtype, float *o_out, int32_t *evicted_pos, void *workspace,
                    size_t workspace_bytes, int *dev_status, kv_stream_t stream) {
  return h2o_decode_steps(q, k_new, v_new, 1, K_cache, V_cache, pos, acc, len, B, Hq, Hkv, cap, d,
                          recent, sink, new_pos, scale, flags, dtype, o_out, evicted_pos, workspace,
                          workspace_bytes, dev_status, stream);
}

int h2o_decode_steps(const void *q, const void *k_new, const void *v_new, int n_steps,
                     void *K_cache, void *V_cache, int32_t *pos, float *acc, int32_t *len, int B,
                     int Hq, int Hkv, int cap, int d, int recent, int sink, int32_t first_pos,
                     float scale, int flags, int dtype, float *o_out, int32_t *evicted_pos,
                     void *workspace, size_t workspace_bytes, int *dev_status,
                     kv_stream_t stream) {
  if (n_steps < 0 || first_pos < 0 || (long long)first_pos + n_steps - 1 > INT_MAX)
    return KV_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || cap <= 0 || recent < 0 || sink < 0 ||
      recent >= cap || !dtype_ok(dtype) || (flags & ~KV_H2O_ALG1) ||
      ((flags & KV_H2O_ALG1) && recent != 0) || !(scale == scale))
    return KV_ERR_INVALID_ARG;
  if (!dim_ok(d)) return KV_ERR_UNSUPPORTED;
  if (!fits((long long)B * Hkv, (long long)cap * d) || !fits((long long)B * Hq, (long long)n_steps * d))
    return KV_ERR_INVALID_ARG;
  if (B == 0 || n_steps == 0) return KV_OK;
  if (!q || !k_new || !v_new || !K_cache || !V_cache || !pos || !acc || !len || !o_out ||
      !evicted_pos)
    return KV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(K_cache) ||
      !aligned16(V_cache))
    return KV_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KV_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < decode_ws_split(B, Hkv, G, cap, d) || !aligned16(workspace))
    return KV_ERR_WORKSPACE;
  return decode_run(q, k_new, v_new, n_steps, K_cache, V_cache, pos, acc, len, B, Hq, Hkv, cap, d,
                    recent, sink, first_pos, scale, flags, dtype, o_out, evicted_pos, workspace,
                    dev_status, static_cast<cudaStream_t>(stream));
}

int h2o_decode_step(const void *q, const void *k_new, const void *v_new, void *K_cache,
                    void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq,
                    int Hkv, int cap, int d, int recent, int32_t new_pos, float scale,
                    int flags, int dtype, float *o_out, int32_t *evicted_pos, void *workspace,
                    size_t workspace_bytes, int *dev_status, kv_stream_t stream) {
  return h2o_decode_step_ex(q, k_new, v_new, K_cache, V_cache, pos, acc, len, B, Hq, Hkv, cap, d,
                            recent, 0, new_pos, scale, flags, dtype, o_out, evicted_pos, workspace,
                            workspace_bytes, dev_status, stream);
}

}  // extern "C"
