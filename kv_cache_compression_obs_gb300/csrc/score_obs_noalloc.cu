// score_obs_noalloc.cu -- kv_score_obs for callers that cannot allocate device memory.
//
// kv_score_obs needs a scratch buffer for the per-row softmax statistics that
// pass between its launches, and takes it from the caller as `workspace`.  Some
// callers have no way to provide one: code embedded in a host framework that
// hands it only its input and output buffers, and code that must not call
// cudaMalloc on its path because the call can synchronise the whole device and
// stall every other stream.  kv_score_obs_noalloc runs the same kernels with the
// scratch taken from a fixed-size array that lives in the library's device
// image instead, so it allocates nothing.
//
// Costs and limits of that array:
//   * KV_SCORE_NOALLOC_SCRATCH_BYTES of device memory on every GPU that loads
//     the library, held until the process exits;
//   * shapes whose scratch need (kv_workspace_size(KV_OP_SCORE_OBS, ...)) is
//     larger are rejected with KV_ERR_WORKSPACE before anything is launched;
//   * every call shares the one array, so calls that overlap on the GPU (two
//     streams, or two host threads) race and corrupt each other's results:
//     serialise them.  The array keeps the last call's contents: every call
//     zeroes the scoring kernels' work-claim counters at its start (an
//     asynchronous memset on the caller's stream, not an allocation), and the
//     kernels write every other entry before they read it.
//   * the device address of the array is looked up (cudaGetSymbolAddress) by
//     the first call on each device, with that device current; make that first
//     call before any stream capture.  The address is cached for the life of
//     the process and is stale after cudaDeviceReset (or any teardown of the
//     primary context): this entry point must not be called after one.
#include <mutex>

#include "kvc_internal.cuh"

namespace {

__device__ __align__(256) unsigned char g_score_scratch[KV_SCORE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_score_scratch on `dev` (the current device); nullptr on failure.
void *scratch_on(int dev) {
  static std::mutex mu;
  static void *addr[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_score_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" int kv_score_obs_noalloc(const void *Q_obs, const void *K, int B, int Hq, int Hkv,
                                    int T, int d, int W, float scale, int dtype, float *s_out,
                                    int *dev_status, kv_stream_t stream) {
  const int rc = kvc::check_score_args(Q_obs, K, B, Hq, Hkv, T, d, W, scale, dtype, s_out);
  if (rc != KV_OK || B == 0) return rc;
  const kvc::ScorePlan plan = kvc::plan_score(B, Hq, Hkv, T, W);
  if (plan.ws_bytes > KV_SCORE_NOALLOC_SCRATCH_BYTES) return KV_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KV_ERR_CUDA;
  void *scratch = scratch_on(dev);
  if (!scratch) return KV_ERR_CUDA;
  return kvc::launch_score_obs(Q_obs, K, B, Hq, Hkv, T, d, W, scale, dtype, s_out, scratch, plan,
                               dev_status, static_cast<cudaStream_t>(stream));
}
