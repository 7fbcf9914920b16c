// kvc_internal.cuh -- shared declarations of the CUDA library (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "kvc.h"

namespace kvc {

constexpr int kNumSmsHint = 152;  // GB300; the launchers query the real count

int device_sm_count();
// Opt a kernel into `bytes` of dynamic shared memory when that plus its static
// shared memory passes 48 KB; nonzero if the device cannot give it.
int ensure_smem(const void *func, size_t bytes);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void count_launches(int n);  // diagnostic counter behind kv_launch_count()
// Remember the CUDA error behind a KV_ERR_CUDA (kv_last_error_detail); returns KV_ERR_CUDA.
int cuda_failure(cudaError_t e, const char *where);
const char *last_detail();

inline int launch_status(int launches = 1) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_failure(e, "kernel launch");
  count_launches(launches);
  return KV_OK;
}

// ---- element access ---------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Unpack one 16-byte vector into floats: 8 bf16 or 4 f32.
template <typename T> struct Vec16;
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4 &v, float *out) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};
template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4 &v, float *out) {
    out[0] = __uint_as_float(v.x);
    out[1] = __uint_as_float(v.y);
    out[2] = __uint_as_float(v.z);
    out[3] = __uint_as_float(v.w);
  }
};

// Host-side argument checks shared by kv_score_obs and kv_score_obs_noalloc:
// KV_OK (with B == 0: nothing to launch) or the status to return.
int check_score_args(const void *Q_obs, const void *K, int B, int Hq, int Hkv, int T, int d,
                     int W, float scale, int dtype, const float *s_out);

// ---- operation plans (shared by the launchers and kv_workspace_size) --------
struct ScorePlan {
  int gw;          // query rows per unit = G * W
  int row_blocks;  // ceil(gw / 64)                          (CUDA-core path)
  int n_splits;    // key splits of the statistics pass      (CUDA-core path)
  int split_len;   // keys per split (multiple of 128)       (CUDA-core path)
  size_t ws_bytes;   // enough for either path
};
ScorePlan plan_score(int B, int Hq, int Hkv, int T, int W);

// Workspace layout of the tensor-core scoring path: claim counters (cleared by
// every call), per-split row statistics, merged row offsets, per-row-block column sums.
struct TcLayout {
  int nrb;        // row blocks of up to 256 query rows per unit
  int ns;         // key splits per row block
  int split_len;  // keys per split (a multiple of 128)
  size_t ctrl_off, part_off, fin_off, pcol_off, bytes;
};
TcLayout tc_layout(int B, int Hq, int Hkv, int T, int W);

struct RefinePlan {
  int chunk;     // elements per entropy chunk
  int n_chunks;  // chunks per head
  size_t beta_offset;  // byte offset of the per-head beta array in the workspace
  size_t ws_bytes;
};
RefinePlan plan_refine(int B, int H, int T);

// ---- launchers (validated arguments only) ------------------------------------
int launch_score_obs(const void *Q, const void *K, int B, int Hq, int Hkv, int T, int d, int W,
                     float scale, int dtype, float *s, void *ws, const ScorePlan &plan,
                     int *status, cudaStream_t st);
int launch_score_combine(const float2 *part, int n_splits, int gw, long rows, float2 *fin,
                         cudaStream_t st);
bool score_tc_eligible(int dtype, int d, int Hq, int Hkv, int W);
int launch_score_obs_tc(const void *Q, const void *K, int B, int Hq, int Hkv, int T, int d, int W,
                        float scale, float *s, void *ws, const ScorePlan &plan, int *status,
                        cudaStream_t st);
int launch_hubkv_refine(const float *s, int B, int H, int T, int pool_width, float gamma,
                        float r, float beta_lo, float beta_hi, int flags, float *z, float *beta,
                        void *ws, const RefinePlan &plan, cudaStream_t st);
int launch_select_topk(const float *z, int B, int H, int T, int k, int recent, int sink,
                       int32_t *idx, cudaStream_t st);
// The refinement's two parts: entropy partials and head weights (into the
// workspace's beta array, copied to beta_out when given), then z.
int launch_refine_beta(const float *s, int B, int H, int T, float beta_lo, float beta_hi, int flags,
                       float *beta_out, void *ws, const RefinePlan &plan, cudaStream_t st);
int launch_refine_apply(const float *s, int B, int H, int T, int half, float gamma, float r, int flags,
                        const float *beta_ws, float *z, cudaStream_t st);
// hubkv_refine then kv_select_topk_ex, z formed inside the selection's load when
// the heads fit on chip; z_tmp ([B][H][T]) is used only when hubkv_select_needs_z.
bool hubkv_select_needs_z(int T, int k, int recent, int sink);
int launch_hubkv_select(const float *s, int B, int H, int T, int pool_width, float gamma, float r,
                        float beta_lo, float beta_hi, int flags, int k, int recent, int sink,
                        int32_t *idx, float *z_out, float *beta_out, void *ws,
                        const RefinePlan &plan, float *z_tmp, cudaStream_t st);
int launch_compact(const void *K, const void *V, const float *s, const int32_t *idx, int B,
                   int H, int T, int k, int d, int dtype, void *K_out, void *V_out, int cap,
                   int32_t *pos, float *acc, int32_t *len, cudaStream_t st);
int launch_select_budget(const float *z, int B, int H, int T, int budget, int floor_k,
                         int recent, int sink, int32_t *idx, int32_t *off, cudaStream_t st);
int launch_compact_ragged(const void *K, const void *V, const float *s, const int32_t *idx,
                          const int32_t *off, int B, int H, int T, int budget, int d, int dtype,
                          void *K_out, void *V_out, int cap, int32_t *pos, float *acc,
                          int32_t *len, int *status, cudaStream_t st);
size_t nested_workspace_bytes(long units, int T, int d, int n_blocks, bool with_a);
int launch_score_nested(const void *K, int B, int H, int T, int d, int dtype, int window,
                        int n_blocks, int n_disc, float lp0, float lp1, float lp2, float thresh,
                        float *score, float *w_out, float *a_out, void *ws, cudaStream_t st);
int launch_decode_step(const void *q, const void *k_new, const void *v_new, void *K_cache,
                       void *V_cache, int32_t *pos, float *acc, int32_t *len, int B, int Hq,
                       int Hkv, int cap, int d, int recent, int sink, int32_t new_pos, float scale,
                       int flags, int dtype, void *workspace, float *o, int32_t *evicted,
                       int *dev_status, cudaStream_t st);
size_t decode_workspace_bytes(long units, int G, int cap, int d);

}  // namespace kvc
