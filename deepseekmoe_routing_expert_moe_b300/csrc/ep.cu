// Expert parallelism: the row bookkeeping of the pages' dispatch / combine
// ("02 · DeepSeek-V3" (PaperTrace) §1.3 node-limited routing, §2 and §5.1:
// experts are partitioned over devices, each token's rows are sent to the
// devices that hold its chosen experts and the outputs come back).
//
// With the experts of a device contiguous (device r holds experts
// [r*El, (r+1)*El)), the expert-sorted dispatch rows of moe_permute are
// already grouped by destination device, so the send side needs no kernel.
// A device receives, from each source device s in order, that source's rows
// for its El experts (expert-sorted within the source's block): the
// "source-major" order.  The grouped GEMM wants the rows of each expert
// together: the "expert-major" order, expert l's rows from source 0, then
// source 1, ...  ep_plan_kernel computes, for every received row i, its
// expert-major position perm[i] and the local segment offsets; the row
// copies in both directions are ep_rows_kernel.
#include <cstdint>

#include "device_common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kPlanThreads = 256;
constexpr int kPlanRowsPerBlock = 1024;

// counts [n_src][n_local]: rows source s sends for local expert l.
// perm[i] for source-major row i = expert-major row; block 0 also writes
// offsets_local [n_local + 1] (expert-major segment starts).
// Exclusive prefix sums of v(0), ..., v(n - 1) into out[0..n) and the total
// into out[n], by all kPlanThreads threads: each takes a contiguous chunk,
// the chunk sums are scanned across the warps, then each chunk is written.
template <class F>
__device__ __forceinline__ void block_exclusive_scan(int n, F v, int* out,
                                                     int* wsum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + kPlanThreads - 1) / kPlanThreads;
  const int a = min(n, tid * per), b = min(n, a + per);
  int loc = 0;
  for (int i = a; i < b; ++i) loc += v(i);
  int incl = loc;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int run = incl - loc, total = 0;
  for (int w = 0; w < kPlanThreads / 32; ++w) {
    run += w < warp ? wsum[w] : 0;
    total += wsum[w];
  }
  for (int i = a; i < b; ++i) {
    out[i] = run;
    run += v(i);
  }
  if (tid == 0) out[n] = total;
  __syncthreads();  // wsum is reused by the next scan
}

__global__ void __launch_bounds__(kPlanThreads)
    ep_plan_kernel(const int32_t* __restrict__ counts, int n_src, int n_local,
                   long long rows, int32_t* __restrict__ perm,
                   int32_t* __restrict__ offsets_local, DevStatus* st) {
  extern __shared__ int sm[];
  __shared__ int wsum[kPlanThreads / 32];
  const int n = n_src * n_local;
  int* src_off = sm;          // [n + 1] exclusive prefix, source-major
  int* exp_off = sm + n + 1;  // [n + 1] exclusive prefix, expert-major (l, s)
  block_exclusive_scan(
      n, [&](int i) { return __ldg(counts + i); }, src_off, wsum);
  block_exclusive_scan(
      n,
      [&](int j) {
        const int l = j / n_src, s = j - l * n_src;
        return __ldg(counts + s * n_local + l);
      },
      exp_off, wsum);
  if (threadIdx.x == 0 && blockIdx.x == 0 && src_off[n] != rows)
    record_error(st, MOE_ERR_DEVICE_BOUNDS, 60);
  if (blockIdx.x == 0) {
    for (int l = threadIdx.x; l <= n_local; l += kPlanThreads)
      offsets_local[l] = l < n_local ? exp_off[l * n_src] : src_off[n];
  }
  const long long lim = min((long long)src_off[n], rows);
  const long long r0 = (long long)blockIdx.x * kPlanRowsPerBlock;
  const long long r1 = min(lim, r0 + kPlanRowsPerBlock);
  for (long long i = r0 + threadIdx.x; i < r1; i += kPlanThreads) {
    // the (source, expert) cell holding source-major row i
    int lo = 0, hi = n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (src_off[mid] <= i)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int s = lo / n_local, l = lo - s * n_local;
    perm[i] = exp_off[l * n_src + s] + (int)(i - src_off[lo]);
  }
  // rows beyond the counts (inconsistent sizes): mapped to themselves
  for (long long i = max(r0, lim) + threadIdx.x;
       i < min(rows, r0 + kPlanRowsPerBlock); i += kPlanThreads)
    perm[i] = (int)i;
}

// inverse = 0: out[perm[i]] = in[i]; inverse = 1: out[i] = in[perm[i]];
// rows of row_bytes bytes in the widest unit that divides them (16-byte
// vectors for bf16 rows and E4M3 codes; 4, 2 or 1 bytes for the rows of
// their scale bytes, H/128 per token), one block per row
template <typename V>
__global__ void __launch_bounds__(128)
    ep_rows_kernel(const uint8_t* __restrict__ in, long long rows,
                   long long row_bytes, const int32_t* __restrict__ perm,
                   int inverse, uint8_t* __restrict__ out, DevStatus* st) {
  const long long i = blockIdx.x;
  const int p = perm[i];
  if (p < 0 || p >= rows) {
    record_error(st, MOE_ERR_DEVICE_BOUNDS, 61);
    return;
  }
  const long long src = inverse ? p : i, dst = inverse ? i : p;
  const V* a = reinterpret_cast<const V*>(in + src * row_bytes);
  V* b = reinterpret_cast<V*>(out + dst * row_bytes);
  for (long long c = threadIdx.x; c < row_bytes / (long long)sizeof(V);
       c += blockDim.x)
    b[c] = __ldg(a + c);
}

}  // namespace

int ep_plan_max_cells() { return 4096; }

cudaError_t launch_ep_plan(const int32_t* counts, int n_src, int n_local,
                           long long rows, int32_t* perm,
                           int32_t* offsets_local, DevStatus* st,
                           cudaStream_t s) {
  const long long nb =
      rows > 0 ? (rows + kPlanRowsPerBlock - 1) / kPlanRowsPerBlock : 1;
  const size_t smem = sizeof(int) * (2 * n_src * n_local + 2);
  ep_plan_kernel<<<(unsigned)nb, kPlanThreads, smem, s>>>(
      counts, n_src, n_local, rows, perm, offsets_local, st);
  return cudaGetLastError();
}

cudaError_t launch_ep_rows(const void* in, long long rows,
                           long long row_bytes, const int32_t* perm,
                           int inverse, void* out, DevStatus* st,
                           cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const uint8_t* a = static_cast<const uint8_t*>(in);
  uint8_t* b = static_cast<uint8_t*>(out);
  if (row_bytes % 16 == 0)
    ep_rows_kernel<uint4><<<(unsigned)rows, 128, 0, s>>>(
        a, rows, row_bytes, perm, inverse, b, st);
  else if (row_bytes % 4 == 0)
    ep_rows_kernel<uint32_t><<<(unsigned)rows, 128, 0, s>>>(
        a, rows, row_bytes, perm, inverse, b, st);
  else if (row_bytes % 2 == 0)
    ep_rows_kernel<uint16_t><<<(unsigned)rows, 128, 0, s>>>(
        a, rows, row_bytes, perm, inverse, b, st);
  else
    ep_rows_kernel<uint8_t><<<(unsigned)rows, 128, 0, s>>>(
        a, rows, row_bytes, perm, inverse, b, st);
  return cudaGetLastError();
}

}  // namespace moe
