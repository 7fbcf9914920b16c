// compact.cu -- "real drop" gather-compaction into a preallocated slot cache
// (H2O page, 两套代码 and FlexGen 改造).
//
//   K_out[m] = K[idx[m]], V_out[m] = V[idx[m]], pos[m] = idx[m], acc[m] = s[idx[m]],
//   len = k, for m < k; slots k..cap-1 are untouched.
// A bit-exact copy: every row moves as whole 16-byte vectors; a warp covers
// 32 consecutive vectors, i.e. 2 rows of 256 bytes (d = 128 bf16), so loads and
// stores are fully coalesced.  Grid: (units x row chunks), each block copying
// kRows rows of K and of V.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int NT = 256;
constexpr int kRows = 64;

__global__ __launch_bounds__(NT) void compact_kernel(
    const uint4 *__restrict__ K, const uint4 *__restrict__ V, const float *__restrict__ s,
    const int32_t *__restrict__ idx, int T, int k, int vpr, int chunks, uint4 *__restrict__ Ko,
    uint4 *__restrict__ Vo, int cap, int32_t *__restrict__ pos, float *__restrict__ acc,
    int32_t *__restrict__ len) {
  const long unit = blockIdx.x / chunks;
  const int m0 = (blockIdx.x % chunks) * kRows;
  const int rows = min(kRows, k - m0);
  const int32_t *iu = idx + unit * (long)k;
  __shared__ int32_t src[kRows];
  if (threadIdx.x < rows) {
    const int j = iu[m0 + threadIdx.x];
    const bool ok = j >= 0 && j < T;  // an out-of-range index leaves its slot untouched
    src[threadIdx.x] = ok ? j : -1;
    if (ok) {
      pos[unit * (long)cap + m0 + threadIdx.x] = j;
      if (acc) acc[unit * (long)cap + m0 + threadIdx.x] = s[unit * (long)T + j];
    }
  }
  if (m0 == 0 && threadIdx.x == 0) len[unit] = k;
  __syncthreads();
  const long in_base = unit * (long)T * vpr;
  const long out_base = (unit * (long)cap + m0) * vpr;
  const int nvec = rows * vpr;
  for (int e = threadIdx.x; e < nvec; e += NT) {
    const int r = e / vpr, v = e - r * vpr;
    if (src[r] < 0) continue;
    const long from = in_base + (long)src[r] * vpr + v;
    const uint4 a = __ldg(K + from);
    const uint4 b = __ldg(V + from);
    Ko[out_base + e] = a;
    Vo[out_base + e] = b;
  }
}

}  // namespace

int launch_compact(const void *K, const void *V, const float *s, const int32_t *idx, int B,
                   int H, int T, int k, int d, int dtype, void *K_out, void *V_out, int cap,
                   int32_t *pos, float *acc, int32_t *len, cudaStream_t st) {
  const long units = (long)B * H;
  const int row_bytes = d * (dtype == KV_BF16 ? 2 : 4);
  const int vpr = row_bytes / 16;
  const int chunks = (k + kRows - 1) / kRows;
  compact_kernel<<<(unsigned)(units * chunks), NT, 0, st>>>(
      static_cast<const uint4 *>(K), static_cast<const uint4 *>(V), s, idx, T, k, vpr, chunks,
      static_cast<uint4 *>(K_out), static_cast<uint4 *>(V_out), cap, pos, (s ? acc : nullptr),
      len);
  return launch_status();
}

}  // namespace kvc
