// compact.cu -- "real drop" gather-compaction into a preallocated slot cache
// (H2O page, 两套代码 and FlexGen 改造).
//
//   K_out[m] = K[idx[m]], V_out[m] = V[idx[m]], pos[m] = idx[m], acc[m] = s[idx[m]],
//   len = k, for m < k; slots k..cap-1 are untouched.
// A bit-exact copy: every row moves as whole 16-byte vectors; a warp covers
// 32 consecutive vectors, i.e. 2 rows of 256 bytes (d = 128 bf16), so loads and
// stores are fully coalesced.  Grid: (units x row chunks), each block copying
// kRows rows of K and of V.
//
// The ragged form takes the CSR output of the layer-level budget (NestedKV
// technical summary, 3. Hoofd-gewijze Geheugentoewijzing): head h of row b keeps
// idx[b][off[b][h] .. off[b][h+1]-1] into its slots 0..n-1 and len = n.  Its
// grid walks the CSR entries themselves (rows x entry chunks), so no block idles
// on a head that keeps few rows; each entry finds its head by a binary search
// over the row's offsets in shared memory.
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

constexpr int kMaxHeadsRagged = 256;

__device__ __forceinline__ void flag_status(int *status, int code) {
  if (status) atomicExch(status, code);
}

__global__ __launch_bounds__(NT) void compact_ragged_kernel(
    const uint4 *__restrict__ K, const uint4 *__restrict__ V, const float *__restrict__ s,
    const int32_t *__restrict__ idx, const int32_t *__restrict__ off, int H, int T, int budget,
    int vpr, int chunks, uint4 *__restrict__ Ko, uint4 *__restrict__ Vo, int cap,
    int32_t *__restrict__ pos, float *__restrict__ acc, int32_t *__restrict__ len,
    int *status) {
  const long row = blockIdx.x / chunks;
  const int e0 = (blockIdx.x % chunks) * kRows;
  __shared__ int32_t so[kMaxHeadsRagged + 1];
  __shared__ long dst[kRows];  // destination slot (unit * cap + m), -1 = skip
  __shared__ long src[kRows];  // source row (unit * T + j)
  __shared__ int row_ok;
  for (int h = threadIdx.x; h <= H; h += NT) so[h] = off[row * (H + 1) + h];
  if (threadIdx.x == 0) row_ok = 1;
  __syncthreads();
  for (int h = threadIdx.x; h <= H; h += NT) {
    const bool bad = (h == 0) ? (so[0] < 0) : (so[h] < so[h - 1] || (h == H && so[H] > budget));
    if (bad) row_ok = 0;
  }
  __syncthreads();
  if (!row_ok) {  // malformed offsets: the whole row stays untouched
    if (e0 == 0 && threadIdx.x == 0) flag_status(status, KV_ERR_INVALID_ARG);
    return;
  }
  if (e0 == 0) {
    for (int h = threadIdx.x; h < H; h += NT) {
      const int n = so[h + 1] - so[h];
      if (n <= cap) len[row * H + h] = n;
      else flag_status(status, KV_ERR_INVALID_ARG);  // that head stays untouched
    }
  }
  const int rows = min(kRows, budget - e0);
  if (threadIdx.x < kRows) {
    long d = -1, f = 0;
    const int e = e0 + threadIdx.x;
    if (threadIdx.x < rows && e >= so[0] && e < so[H]) {
      int a = 0, b = H - 1;  // the head h with so[h] <= e < so[h + 1]
      while (a < b) {
        const int mid = (a + b) >> 1;
        if (so[mid + 1] <= e) a = mid + 1;
        else b = mid;
      }
      const int n = so[a + 1] - so[a];
      const int j = idx[row * (long)budget + e];
      if (n <= cap && j >= 0 && j < T) {  // out-of-range indexes leave the slot untouched
        const long unit = row * H + a;
        const int m = e - so[a];
        d = unit * cap + m;
        f = unit * (long)T + j;
        pos[d] = j;
        if (acc) acc[d] = s[f];
      }
    }
    dst[threadIdx.x] = d;
    src[threadIdx.x] = f;
  }
  __syncthreads();
  const int nvec = rows * vpr;
  for (int e = threadIdx.x; e < nvec; e += NT) {
    const int r = e / vpr, v = e - r * vpr;
    if (dst[r] < 0) continue;
    const long from = src[r] * vpr + v;
    const uint4 a = __ldg(K + from);
    const uint4 b = __ldg(V + from);
    Ko[dst[r] * vpr + v] = a;
    Vo[dst[r] * vpr + v] = b;
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

int launch_compact_ragged(const void *K, const void *V, const float *s, const int32_t *idx,
                          const int32_t *off, int B, int H, int T, int budget, int d, int dtype,
                          void *K_out, void *V_out, int cap, int32_t *pos, float *acc,
                          int32_t *len, int *status, cudaStream_t st) {
  const int row_bytes = d * (dtype == KV_BF16 ? 2 : 4);
  const int vpr = row_bytes / 16;
  const int chunks = budget > 0 ? (budget + kRows - 1) / kRows : 1;
  compact_ragged_kernel<<<(unsigned)((long)B * chunks), NT, 0, st>>>(
      static_cast<const uint4 *>(K), static_cast<const uint4 *>(V), s, idx, off, H, T, budget,
      vpr, chunks, static_cast<uint4 *>(K_out), static_cast<uint4 *>(V_out), cap, pos,
      (s ? acc : nullptr), len, status);
  return launch_status();
}

}  // namespace kvc
