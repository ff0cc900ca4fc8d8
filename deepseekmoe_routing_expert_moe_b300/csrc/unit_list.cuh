// Work units of the persistent grouped expert GEMMs (BF16 in
// grouped_gemm.cu, FP8 with power-of-two scales in mx_gemm.cu) and the
// epilogue helpers they share.
//
// The token rows are grouped in segments: segment 0 is the shared expert
// over all T tokens, segment 1 + e the rows [offsets[e], offsets[e+1]) of
// routed expert e.  A unit is (segment, feature block f, chunk of the
// segment's rows); segments longer than NT rows are cut into equal chunks
// rounded up to 16 rows.  `useg` is the exclusive prefix of the units per
// segment (useg[NS] = total), `srow0` / `srows` the segments' first row and
// row count, all in shared memory.
#pragma once

#include <cstdint>

#include "device_common.cuh"

namespace moe {

// One unit of work, decoded identically by every role.
struct Unit {
  int seg;    // 0 = shared expert, 1 + e = routed expert e
  int f;      // feature block
  int row0;   // first row of the chunk in the token / output tensors
  int rows;   // valid rows in the chunk (1..NT of the pipeline shape)
  int n;      // MMA N: rows rounded up to 16
};

__device__ __forceinline__ int round16(int v) { return (v + 15) & ~15; }

// Segment tables in shared memory: srow0/srows per segment, useg the
// exclusive prefix of units per segment (useg[NS] = total).
template <int NT>
__device__ __forceinline__ Unit decode_unit(int u, const int* useg,
                                            const int* srow0,
                                            const int* srows, int NS) {
  int lo = 0, hi = NS - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (useg[mid] <= u)
      lo = mid;
    else
      hi = mid - 1;
  }
  Unit x;
  x.seg = lo;
  const int R = srows[lo];
  const int nch = (R + NT - 1) / NT;
  const int cs = round16((R + nch - 1) / nch);
  const int local = u - useg[lo];
  x.f = local / nch;
  const int c = local - x.f * nch;
  x.row0 = srow0[lo] + c * cs;
  x.rows = min(cs, R - c * cs);
  x.n = round16(x.rows);
  return x;
}

// silu(g) = g / (1 + e^-g).  The exponent's argument is capped at 80 so
// that 1 + e stays below 2^116, inside the documented range of the fast
// division, for every g: below g = -80 the true value is under 1e-33 in
// magnitude and the capped form returns g / (1 + e^80), also under 1e-33
// (a NaN g stays NaN).
__device__ __forceinline__ float silu_f(float g) {
  return __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f)));
}

// Columns [0, n) of this thread's TMEM lane (accumulator at `taddr`),
// rounded to bf16 pairs: pk[j / 2] holds column j in its low (even j) or
// high (odd j) half.  COLS bounds n at compile time so pk stays in
// registers.
template <int COLS>
__device__ __forceinline__ void load_packed(uint32_t taddr, int n,
                                            uint32_t (&pk)[COLS / 2]) {
#pragma unroll
  for (int c = 0; c < COLS / 16; ++c) {
    if (16 * c < n) {
      uint32_t v[16];
      tmem_ld16(taddr + 16 * c, v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 8; ++i)
        pk[8 * c + i] = pack_bf16x2(__uint_as_float(v[2 * i]),
                                    __uint_as_float(v[2 * i + 1]));
    }
  }
}

// out[j * ld] = column j of pk for j < rows (one bf16 per token row).
template <int COLS>
__device__ __forceinline__ void store_packed(const uint32_t (&pk)[COLS / 2],
                                             uint16_t* out, int ld,
                                             int rows) {
#pragma unroll
  for (int c = 0; c < COLS / 16; ++c) {
    if (16 * c < rows) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (16 * c + i < rows)
          out[(size_t)(16 * c + i) * ld] = static_cast<uint16_t>(
              (i & 1) ? (pk[8 * c + i / 2] >> 16)
                      : (pk[8 * c + i / 2] & 0xFFFFu));
      }
    }
  }
}

}  // namespace moe
