// FP8 (E4M3) fine-grained quantization ("02 · DeepSeek-V3" §2, mixed
// precision): activations in 1 x 128 tiles (one row, 128 channels),
// weights in 128 x 128 blocks, one fp32 scale per group from the group's
// own max |value| taken online:
//   s = amax / 448 (correctly rounded; 1 for an all-zero group)
//   code = E4M3(x / s), the fp32 quotient rounded to nearest even and
//          saturated to +-448 (cvt.rn.satfinite)
// so every code is decided from the same fp32 values as the CPU oracle's.
// The power-of-two variant (the microscaling form the same section points
// to for Blackwell's tensor cores) takes s = 2^e, e the least exponent with
// 448 * 2^e >= amax, stores e + 127 as one byte (UE8M0) and codes
// E4M3(x * 2^-e) -- an exact product, so the code is the E4M3 rounding of
// the exact quotient.
#include <cuda_fp8.h>

#include <cstdint>

#include "device_common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr float kE4m3Max = 448.0f;

// A group's scale, from its max |value|: the fp32 scale amax / 448 ...
struct ScaleF32 {
  using T = float;
  float s;
  __device__ explicit ScaleF32(float amax) {
    s = amax > 0.0f ? __fdiv_rn(amax, kE4m3Max) : 1.0f;
  }
  __device__ uint32_t code(float v) const {
    return (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(v, s), __NV_SATFINITE,
                                           __NV_E4M3);
  }
  __device__ T stored() const { return s; }
};

// ... or the power-of-two scale 2^e, stored as the byte e + 127
struct ScaleE8 {
  using T = uint8_t;
  int e;
  float inv;  // 2^-e
  __device__ explicit ScaleE8(float amax) {
    e = ue8m0_exponent(amax);
    inv = pow2_neg(e);
  }
  __device__ uint32_t code(float v) const {
    return (uint32_t)__nv_cvt_float_to_fp8(v * inv, __NV_SATFINITE,
                                           __NV_E4M3);
  }
  __device__ T stored() const { return (uint8_t)(e + 127); }
};

// four codes, first value in the lowest byte (memory order)
template <class S>
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c,
                                           float d, const S& s) {
  return s.code(a) | (s.code(b) << 8) | (s.code(c) << 16) |
         (s.code(d) << 24);
}

// ------------------------------------------------------------------
// 1 x 128 tiles: one warp per (row, group of up to kTilesPerWarp tiles), 4
// consecutive values per lane; the group's loads are all issued before the
// first tile is reduced, and the token's dispatch rows are read once per
// group (lane k < K holds dest[r*K + k]).  q[r] (if q != NULL) and, with
// dest != NULL, the dispatch copies qp[dest[r*K + k]] for k < K (K <= 32)
// receive the codes; s / sp the scales.
// ------------------------------------------------------------------
constexpr int kRowsWarps = 8;
constexpr int kTilesPerWarp = 8;

template <class S>
__global__ void __launch_bounds__(kRowsWarps * 32)
    quant_rows_kernel(const uint16_t* __restrict__ x, long long R, int C,
                      const int32_t* __restrict__ dest, int K, long long RK,
                      uint8_t* __restrict__ q, typename S::T* __restrict__ s,
                      uint8_t* __restrict__ qp,
                      typename S::T* __restrict__ sp, DevStatus* st) {
  const int lane = threadIdx.x & 31;
  const int tiles = C / 128;
  const int groups = (tiles + kTilesPerWarp - 1) / kTilesPerWarp;
  const long long g =
      (long long)blockIdx.x * kRowsWarps + (threadIdx.x >> 5);
  if (g >= R * groups) return;
  const long long r = g / groups;
  const int t0 = (int)(g - r * groups) * kTilesPerWarp;
  int dr_mine = 0;
  bool ok_mine = false;
  if (dest != nullptr && lane < K) {
    dr_mine = __ldg(dest + (size_t)r * K + lane);
    ok_mine = dr_mine >= 0 && dr_mine < RK;
    if (!ok_mine && t0 == 0) record_error(st, MOE_ERR_DEVICE_BOUNDS, 40);
  }
  uint2 raw[kTilesPerWarp];
#pragma unroll
  for (int i = 0; i < kTilesPerWarp; ++i)
    if (t0 + i < tiles)
      raw[i] = __ldg(reinterpret_cast<const uint2*>(
          x + (size_t)r * C + (size_t)(t0 + i) * 128 + lane * 4));
#pragma unroll
  for (int i = 0; i < kTilesPerWarp; ++i) {
    const int tile = t0 + i;
    if (tile >= tiles) break;
    const float v0 = bf16_lo(raw[i].x), v1 = bf16_hi(raw[i].x);
    const float v2 = bf16_lo(raw[i].y), v3 = bf16_hi(raw[i].y);
    const float m = fmaxf(fmaxf(fabsf(v0), fabsf(v1)),
                          fmaxf(fabsf(v2), fabsf(v3)));
    // |v| bit patterns order like the values (non-negative floats)
    const float amax =
        __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));
    const S sc(amax);
    const uint32_t code = e4m3x4(v0, v1, v2, v3, sc);
    const size_t off = (size_t)tile * 128 + lane * 4;
    if (q != nullptr) {
      *reinterpret_cast<uint32_t*>(q + (size_t)r * C + off) = code;
      if (lane == 0) s[(size_t)r * tiles + tile] = sc.stored();
    }
    if (dest != nullptr) {
      for (int k = 0; k < K; ++k) {
        const int dr = __shfl_sync(0xffffffffu, dr_mine, k);
        if (!__shfl_sync(0xffffffffu, ok_mine, k)) continue;
        *reinterpret_cast<uint32_t*>(qp + (size_t)dr * C + off) = code;
        if (lane == 0) sp[(size_t)dr * tiles + tile] = sc.stored();
      }
    }
  }
}

// ------------------------------------------------------------------
// 128 x 128 blocks: one 256-thread CTA per block; thread i holds rows
// {i/16 + 16 j : j < 8}, columns (i % 16) * 8 .. +8 of the block (64
// values), so a warp reads two full 256-byte row segments per step.
// ------------------------------------------------------------------
template <class S>
__global__ void __launch_bounds__(256)
    quant_blocks_kernel(const uint16_t* __restrict__ w, int C,
                        uint8_t* __restrict__ q,
                        typename S::T* __restrict__ s) {
  __shared__ float wmax[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bc = blockIdx.x, br = blockIdx.y, nbc = gridDim.x;
  const int c0 = bc * 128 + (tid & 15) * 8;
  const size_t r0 = (size_t)br * 128 + (tid >> 4);
  float v[8][8];
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 raw =
        __ldg(reinterpret_cast<const uint4*>(w + (r0 + 16 * j) * C + c0));
    const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[j][2 * i] = bf16_lo(u[i]);
      v[j][2 * i + 1] = bf16_hi(u[i]);
      m = fmaxf(m, fmaxf(fabsf(v[j][2 * i]), fabsf(v[j][2 * i + 1])));
    }
  }
  const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
  if (lane == 0) wmax[warp] = __uint_as_float(wm);
  __syncthreads();
  float amax = wmax[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, wmax[i]);
  const S sc(amax);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint2 o;
    o.x = e4m3x4(v[j][0], v[j][1], v[j][2], v[j][3], sc);
    o.y = e4m3x4(v[j][4], v[j][5], v[j][6], v[j][7], sc);
    *reinterpret_cast<uint2*>(q + (r0 + 16 * j) * C + c0) = o;
  }
  if (tid == 0) s[(size_t)br * nbc + bc] = sc.stored();
}

template <class S>
cudaError_t quant_rows(const uint16_t* x, long long R, int C,
                       const int32_t* dest, int K, uint8_t* q,
                       typename S::T* s, uint8_t* qp, typename S::T* sp,
                       DevStatus* st, cudaStream_t stream) {
  const long long warps =
      R * ((C / 128 + kTilesPerWarp - 1) / kTilesPerWarp);
  if (warps == 0) return cudaSuccess;
  const long long blocks = (warps + kRowsWarps - 1) / kRowsWarps;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  quant_rows_kernel<S><<<(unsigned)blocks, kRowsWarps * 32, 0, stream>>>(
      x, R, C, dest, K, R * K, q, s, qp, sp, st);
  return cudaGetLastError();
}

template <class S>
cudaError_t quant_blocks(const uint16_t* w, long long R, int C, uint8_t* q,
                         typename S::T* s, cudaStream_t stream) {
  if (R == 0) return cudaSuccess;
  if (R / 128 > 65535) return cudaErrorInvalidValue;
  quant_blocks_kernel<S><<<dim3(C / 128, (unsigned)(R / 128)), 256, 0,
                           stream>>>(w, C, q, s);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_rows(const uint16_t* x, long long R, int C,
                              const int32_t* dest, int K, uint8_t* q,
                              float* s, uint8_t* qp, float* sp,
                              DevStatus* st, cudaStream_t stream) {
  return quant_rows<ScaleF32>(x, R, C, dest, K, q, s, qp, sp, st, stream);
}

cudaError_t launch_quant_blocks(const uint16_t* w, long long R, int C,
                                uint8_t* q, float* s, cudaStream_t stream) {
  return quant_blocks<ScaleF32>(w, R, C, q, s, stream);
}

cudaError_t launch_quant_rows_e8(const uint16_t* x, long long R, int C,
                                 const int32_t* dest, int K, uint8_t* q,
                                 uint8_t* s, uint8_t* qp, uint8_t* sp,
                                 DevStatus* st, cudaStream_t stream) {
  return quant_rows<ScaleE8>(x, R, C, dest, K, q, s, qp, sp, st, stream);
}

cudaError_t launch_quant_blocks_e8(const uint16_t* w, long long R, int C,
                                   uint8_t* q, uint8_t* s,
                                   cudaStream_t stream) {
  return quant_blocks<ScaleE8>(w, R, C, q, s, stream);
}

}  // namespace moe
