// Routing, dispatch order, gather, combine and the bias step of the
// DeepSeekMoE layer ("02 · DeepSeek-V3" (PaperTrace) §1.3, §1.4; dispatch
// and combine as in §2 / §5.1).  These are HBM- or latency-bound SIMT
// kernels; the expert GEMMs live in grouped_gemm.cu.
#include <cfloat>
#include <algorithm>
#include <climits>
#include <cstdint>

#include "device_common.cuh"
#include "internal.h"

namespace moe {

// ===================================================================
// Router logits: z[t, e] = sum_h x[t, h] * W_r[e, h], fp32 FMA chain in h
// order per output.  64x64 output tile per 256-thread block, 4x4 outputs
// per thread, K staged through shared memory 32 at a time.
// ===================================================================
namespace {
constexpr int RL_BM = 64, RL_BN = 64, RL_BK = 32;

__global__ void __launch_bounds__(256)
    router_logits_kernel(const uint16_t* __restrict__ x,
                         const float* __restrict__ w,
                         const float* __restrict__ offset,
                         float* __restrict__ z, int T, int H, int E) {
  __shared__ float xs[RL_BK][RL_BM + 4];
  __shared__ float ws[RL_BK][RL_BN + 4];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * RL_BM, e0 = blockIdx.y * RL_BN;
  const int ty = tid / 16, tx = tid % 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += RL_BK) {
    {  // x tile: 64 rows x 32 bf16 = 256 x 16 B
      const int r = tid / 4, c = (tid % 4) * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t0 + r < T)
        v = *reinterpret_cast<const uint4*>(x + (size_t)(t0 + r) * H + k0 + c);
      const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xs[c + 2 * i][r] = bf16_lo(q[i]);
        xs[c + 2 * i + 1][r] = bf16_hi(q[i]);
      }
    }
#pragma unroll
    for (int p = 0; p < 2; ++p) {  // w tile: 64 rows x 32 fp32 = 512 x 16 B
      const int li = tid + p * 256;
      const int r = li / 8, c = (li % 8) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e0 + r < E)
        v = *reinterpret_cast<const float4*>(w + (size_t)(e0 + r) * H + k0 + c);
      ws[c][r] = v.x;
      ws[c + 1][r] = v.y;
      ws[c + 2][r] = v.z;
      ws[c + 3][r] = v.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < RL_BK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[k][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ws[k][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E)
        z[(size_t)t * E + e] =
            offset != nullptr ? acc[i][j] + offset[e] : acc[i][j];
    }
  }
}
}  // namespace

// Exact split of the fp32 router weight into three bf16 parts:
//   hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid),
// each subtraction exact in fp32, so hi + mid + lo == w for every normal w
// (8 + 8 + 8 significant bits cover fp32's 24).  Layout [3, E, H].
__global__ void split_router_weight_kernel(const float* __restrict__ w,
                                           size_t n,
                                           uint16_t* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const float v = w[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    out[i] = __bfloat16_as_ushort(hi);
    out[n + i] = __bfloat16_as_ushort(mid);
    out[2 * n + i] = __bfloat16_as_ushort(lo);
  }
}

cudaError_t launch_split_router_weight(const float* w, int E, int H,
                                       uint16_t* w_split, cudaStream_t s) {
  const size_t n = (size_t)E * H;
  const int blocks = (int)std::min<size_t>((n + 255) / 256, 4 * 148);
  split_router_weight_kernel<<<blocks, 256, 0, s>>>(w, n, w_split);
  return cudaGetLastError();
}

cudaError_t launch_router_logits(const uint16_t* x, const float* w_router,
                                 const float* offset, float* logits, int T,
                                 int H, int E, cudaStream_t s) {
  dim3 grid((T + RL_BM - 1) / RL_BM, (E + RL_BN - 1) / RL_BN);
  router_logits_kernel<<<grid, 256, 0, s>>>(x, w_router, offset, logits, T,
                                            H, E);
  return cudaGetLastError();
}

// ===================================================================
// fp32 sigmoid, one fixed sequence of correctly rounded IEEE operations so
// that selection is reproducible bit for bit on any conforming machine:
//   w = min(max(-z, -32), 80); n = rint(w * log2 e)
//   r = (w - n*LN2_HI) - n*LN2_LO     (Cody & Waite split of ln 2)
//   p = Horner of sum_{k<=7} r^k / k!, one rounded multiply and one
//       rounded add per step (explicit _rn intrinsics: never contracted)
//   s = 1 / (1 + p * 2^n)
// Constants, derived from the mathematics: LN2_HI = ln 2 rounded to 16
// significant bits (so n*LN2_HI is exact for |n| < 2^8), LN2_LO = the fp32
// rounding of ln 2 - LN2_HI, log2 e and 1/k! rounded to fp32.  For w < -32
// the term 2^-46 vanishes against 1, so the lower clamp changes no result;
// the upper one keeps p * 2^n a normal number.
// ===================================================================
__device__ __forceinline__ float sigmoid_f32(float z) {
  constexpr float kLog2e = 0x1.715476p+0f;
  constexpr float kLn2Hi = 0x1.62e4p-1f;
  constexpr float kLn2Lo = 0x1.7f7d1cp-20f;
  constexpr float kC7 = 0x1.a01a02p-13f;  // 1/5040
  constexpr float kC6 = 0x1.6c16c2p-10f;  // 1/720
  constexpr float kC5 = 0x1.111112p-7f;   // 1/120
  constexpr float kC4 = 0x1.555556p-5f;   // 1/24
  constexpr float kC3 = 0x1.555556p-3f;   // 1/6
  const float w = fminf(fmaxf(-z, -32.0f), 80.0f);
  const float n = rintf(__fmul_rn(w, kLog2e));
  const float r = __fsub_rn(__fsub_rn(w, __fmul_rn(n, kLn2Hi)),
                            __fmul_rn(n, kLn2Lo));
  float p = kC7;
  p = __fadd_rn(__fmul_rn(p, r), kC6);
  p = __fadd_rn(__fmul_rn(p, r), kC5);
  p = __fadd_rn(__fmul_rn(p, r), kC4);
  p = __fadd_rn(__fmul_rn(p, r), kC3);
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  const float two_n = __int_as_float((static_cast<int>(n) + 127) << 23);
  const float e = __fmul_rn(p, two_n);
  // the correctly rounded reciprocal: the same value as 1 / (1 + e)
  return __frcp_rn(__fadd_rn(1.0f, e));
}

// order-preserving map fp32 -> uint32 (larger float -> larger key)
__device__ __forceinline__ uint32_t f32_order_key(float v) {
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ===================================================================
// Routing: one warp per token.  Lane l holds experts [l*EPL, (l+1)*EPL);
// expert groups are whole lane ranges of LPG lanes (LPG a power of 2), so
// the group top-2 is a lane-local top-2 plus an xor butterfly.
//   u = s + b                      selection score (eq. 16)
//   S_g = top1 + top2 of u in g    group score (§1.3)
//   kept = rank of (S_g desc, g asc) < topk_group
//   slots: the topk largest (u desc, e asc) among the kept groups' experts
//   gate_k = s_k / (s_0 + ... + s_{K-1}) summed in slot order (eq. 13)
// Selection: every lane sorts its EPL candidates once (Batcher's odd-even
// merge network on a 64-bit key: the order-preserving bits of u above ~e,
// so the key order is (u desc, e asc) and all keys are distinct; experts of
// dropped groups get u-bits 0, below every kept expert) into shared memory.
// Each of the topk rounds then compares only the lanes' list heads -- one
// warp max of the u-bits, one of the ~e bits among the lanes holding that
// maximum -- and the winning lane advances its head.  The block's
// per-expert histogram is accumulated in shared memory with integer atomics
// and written as one row of block_counts.
// ===================================================================
namespace {

template <int EPL>
__device__ __forceinline__ void load_row(const float* __restrict__ p,
                                         float (&v)[EPL]) {
  if constexpr (EPL % 4 == 0) {
#pragma unroll
    for (int j = 0; j < EPL; j += 4) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(p + j));
      v[j] = q.x;
      v[j + 1] = q.y;
      v[j + 2] = q.z;
      v[j + 3] = q.w;
    }
  } else if constexpr (EPL == 2) {
    const float2 q = __ldg(reinterpret_cast<const float2*>(p));
    v[0] = q.x;
    v[1] = q.y;
  } else {
    v[0] = __ldg(p);
  }
}

// descending compare-exchange of two distinct 64-bit keys
__device__ __forceinline__ void cx_desc(uint64_t& a, uint64_t& b) {
  const uint64_t hi = a > b ? a : b;
  const uint64_t lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// Batcher's odd-even merge sort of N (a power of 2) keys, descending; all
// indices are compile-time constants once the loops are unrolled, so the
// keys stay in registers (19 compare-exchanges for N = 8)
template <int N>
__device__ __forceinline__ void sort_desc(uint64_t (&k)[N]) {
#pragma unroll
  for (int p = 1; p < N; p <<= 1) {
#pragma unroll
    for (int q = p; q >= 1; q >>= 1) {
#pragma unroll
      for (int j = q % p; j <= N - 1 - q; j += 2 * q) {
#pragma unroll
        for (int i = 0; i < q; ++i) {
          if (i + j + q < N && (i + j) / (2 * p) == (i + j + q) / (2 * p))
            cx_desc(k[i + j], k[i + j + q]);
        }
      }
    }
  }
}

// A plain load of shared memory the calling thread wrote earlier, kept as
// a load: the sorted lists are written from registers that the sorting
// network permuted, and the compiler is not to substitute a register for
// this dynamically indexed read.
__device__ __forceinline__ uint64_t ld_shared_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

// shared memory of one warp: the sorted candidate lists, entry h of lane l
// at [h][l] (a warp's stores of one h are consecutive), then s by expert
template <int EPL>
struct RouteWarpSmem {
  static constexpr int KEY_BYTES = EPL * 32 * 8;
  static constexpr int BYTES = KEY_BYTES + EPL * 32 * 4;
};

template <int EPL, int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
    route_kernel(const float* __restrict__ logits,
                 const float* __restrict__ bias, int T, int E, int G, int M,
                 int K, int LPG, int32_t* __restrict__ topk_idx,
                 float* __restrict__ topk_gate,
                 int32_t* __restrict__ block_counts) {
  __shared__ int cnt[1024];
  extern __shared__ __align__(16) uint8_t route_smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* skey = reinterpret_cast<uint64_t*>(
      route_smem + warp * RouteWarpSmem<EPL>::BYTES);
  float* ss = reinterpret_cast<float*>(
      route_smem + warp * RouteWarpSmem<EPL>::BYTES +
      RouteWarpSmem<EPL>::KEY_BYTES);
  for (int i = tid; i < E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();

  const int lanes_used = E / EPL;
  const bool active = lane < lanes_used;
  const int my_g = lane / LPG;
  float b[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) b[j] = active ? bias[lane * EPL + j] : 0.f;

  // this block's tokens (the grid has route_blocks(T) blocks)
  const int tok0 = route_block_start(blockIdx.x, T, gridDim.x);
  const int tok1 = route_block_start(blockIdx.x + 1, T, gridDim.x);
  for (int tt = warp; tt < kRouteTokensPerBlock; tt += WARPS) {
    const int t = tok0 + tt;
    if (t >= tok1) break;
    float s[EPL], u[EPL];
    if (active) {
      load_row<EPL>(logits + (size_t)t * E + lane * EPL, s);
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        s[j] = sigmoid_f32(s[j]);
        u[j] = __fadd_rn(s[j], b[j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        s[j] = 0.f;
        u[j] = -INFINITY;
      }
    }
    // ---- group score: two largest u of the group (a multiset)
    float a1 = -INFINITY, a2 = -INFINITY;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      if (u[j] > a1) {
        a2 = a1;
        a1 = u[j];
      } else if (u[j] > a2) {
        a2 = u[j];
      }
    }
    for (int off = 1; off < LPG; off <<= 1) {
      const float o1 = __shfl_xor_sync(0xffffffffu, a1, off);
      const float o2 = __shfl_xor_sync(0xffffffffu, a2, off);
      const float n2 = fmaxf(fminf(a1, o1), fmaxf(a2, o2));
      a1 = fmaxf(a1, o1);
      a2 = n2;
    }
    const float S = __fadd_rn(a1, a2);
    // ---- kept groups: rank by (S desc, g asc)
    int rank = 0;
    for (int g = 0; g < G; ++g) {
      const float Sg = __shfl_sync(0xffffffffu, S, g * LPG);
      rank += (Sg > S) || (Sg == S && g < my_g);
    }
    const bool kept = active && my_g < G && rank < M;
    // ---- this lane's candidates, sorted once by (u desc, e asc)
    uint64_t key[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const uint32_t hi = kept ? f32_order_key(u[j]) : 0u;
      key[j] = (static_cast<uint64_t>(hi) << 32) |
               static_cast<uint32_t>(~(lane * EPL + j));
    }
    sort_desc<EPL>(key);
#pragma unroll
    for (int j = 0; j < EPL; ++j) skey[j * 32 + lane] = key[j];
    if (active) {
#pragma unroll
      for (int j = 0; j < EPL; ++j) ss[lane * EPL + j] = s[j];
    }
    __syncwarp();
    // ---- top-K: K rounds over the lane heads
    uint64_t head = key[0];
    int h = 0;
    float den = 0.f, my_s = 0.f;
    int my_e = 0;
    for (int k = 0; k < K; ++k) {
      const uint32_t khi = static_cast<uint32_t>(head >> 32);
      const uint32_t mhi = __reduce_max_sync(0xffffffffu, khi);
      const uint32_t klo =
          khi == mhi ? static_cast<uint32_t>(head) : 0u;
      const uint32_t mlo = __reduce_max_sync(0xffffffffu, klo);
      int e = static_cast<int>(~mlo);
      // only a non-finite bias can exhaust the kept candidates: stay in
      // bounds
      if (mhi == 0u || e < 0 || e >= E) e = 0;
      // the lane that won advances its head (every lane reloads its own,
      // branch-free)
      h += (khi == mhi && static_cast<uint32_t>(head) == mlo) ? 1 : 0;
      head = h < EPL ? ld_shared_u64(&skey[h * 32 + lane]) : 0ull;
      const float se = ss[e];
      den = __fadd_rn(den, se);
      if (lane == k) {
        my_e = e;
        my_s = se;
      }
    }
    if (lane < K) {
      topk_idx[(size_t)t * K + lane] = my_e;
      topk_gate[(size_t)t * K + lane] = __fdiv_rn(my_s, den);
      atomicAdd(&cnt[my_e], 1);
    }
    __syncwarp();
  }
  __syncthreads();
  for (int i = tid; i < E; i += blockDim.x)
    block_counts[(size_t)blockIdx.x * E + i] = cnt[i];
}

// ===================================================================
// Sequence-wise balance loss ("02 · DeepSeek-V3" §1.4, eq. 17-20), three
// deterministic passes:
//   1. one warp per token: s = sigmoid(z) (the routing sigmoid, so the
//      top-K decision matches the oracle bit for bit), den = sum_j s_j
//      (lane-local in expert order, then an xor butterfly, so every lane
//      holds the same sum), s' = s * (1/den) (one correctly rounded
//      reciprocal per token), and the raw top-K of s over all experts (no
//      bias, no group limit; ties: lower index).  Writes s' [T, E] fp32
//      and the top-K flags [T, E] u8 to the workspace.
//   2. one CTA per (sequence, 32 experts, row split): the split's rows are
//      cut into 32 ranges summed per expert in token order, then the 32
//      range sums added in order.  With one split per sequence it writes
//      P_i = (sum_t s'_{t,i}) / T_s and c_i = sum_t flag_{t,i} directly;
//      with rs > 1 splits (short batches: the grid would not fill the
//      SMs) it writes per-split partial sums.
//   3. one CTA per sequence: the rs partial sums added in split order (when
//      rs > 1), f_i = E c_i / (K T_s), L = alpha sum_i f_i P_i (xor
//      butterfly within a warp, warps added in order).
// ===================================================================
// one token per warp, 8 warps per block: the grid is many small blocks, so
// the SMs receive nearly equal shares of tokens (64-token blocks left some
// SMs with two blocks and others with one at T = 16384)
constexpr int kBalWarps = 8;
constexpr int kBalTokensPerBlock = kBalWarps;

template <int EPL>
__device__ __forceinline__ void store_row(float* __restrict__ p,
                                          const float (&v)[EPL]) {
  if constexpr (EPL % 4 == 0) {
#pragma unroll
    for (int j = 0; j < EPL; j += 4)
      *reinterpret_cast<float4*>(p + j) =
          make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
  } else if constexpr (EPL == 2) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
  } else {
    p[0] = v[0];
  }
}

// flag byte j = bit j of `pick`
template <int EPL>
__device__ __forceinline__ void store_flags(uint8_t* __restrict__ p,
                                            uint32_t pick) {
  if constexpr (EPL % 4 == 0) {
#pragma unroll
    for (int j = 0; j < EPL; j += 4)
      *reinterpret_cast<uint32_t*>(p + j) =
          ((pick >> j) & 1u) | (((pick >> (j + 1)) & 1u) << 8) |
          (((pick >> (j + 2)) & 1u) << 16) | (((pick >> (j + 3)) & 1u) << 24);
  } else {
#pragma unroll
    for (int j = 0; j < EPL; ++j) p[j] = (uint8_t)((pick >> j) & 1u);
  }
}

template <int EPL, int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
    balance_token_kernel(const float* __restrict__ logits, int T, int E,
                         int K, float* __restrict__ sp,
                         uint8_t* __restrict__ flags) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool active = lane < E / EPL;
  const int tok0 = blockIdx.x * kBalTokensPerBlock;
  for (int tt = warp; tt < kBalTokensPerBlock; tt += WARPS) {
    const int t = tok0 + tt;
    if (t >= T) break;
    float s[EPL];
    if (active) {
      load_row<EPL>(logits + (size_t)t * E + lane * EPL, s);
#pragma unroll
      for (int j = 0; j < EPL; ++j) s[j] = sigmoid_f32(s[j]);
    } else {
#pragma unroll
      for (int j = 0; j < EPL; ++j) s[j] = 0.f;
    }
    float den = 0.f;
#pragma unroll
    for (int j = 0; j < EPL; ++j) den = __fadd_rn(den, s[j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      den = __fadd_rn(den, __shfl_xor_sync(0xffffffffu, den, off));
    // raw top-K of s by (s desc, e asc)
    float cu[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) cu[j] = active ? s[j] : -INFINITY;
    uint32_t pick = 0;
    for (int k = 0; k < K; ++k) {
      float bv = -INFINITY;
      int bj = 0;
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        if (cu[j] > bv) {
          bv = cu[j];
          bj = j;
        }
      }
      const uint32_t key = f32_order_key(bv);
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
      const int cand = (key == kmax && bv != -INFINITY) ? lane * EPL + bj
                                                        : INT_MAX;
      const int e = __reduce_min_sync(0xffffffffu, cand);
      if (e == INT_MAX) break;  // fewer than K finite scores: cannot happen
      if (lane == e / EPL) {
        const int oj = e - lane * EPL;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
          if (j == oj) {
            cu[j] = -INFINITY;
            pick |= 1u << j;
          }
        }
      }
    }
    if (active) {
      const float rden = __frcp_rn(den);
      float o[EPL];
#pragma unroll
      for (int j = 0; j < EPL; ++j) o[j] = __fmul_rn(s[j], rden);
      store_row<EPL>(sp + (size_t)t * E + lane * EPL, o);
      store_flags<EPL>(flags + (size_t)t * E + lane * EPL, pick);
    }
  }
}

// tokens [a, b) of sequence q
__device__ __forceinline__ void seq_range(int q, int S, int T, int& a,
                                          int& b) {
  const long long a64 = (long long)q * S;
  a = (int)a64;
  b = (int)min((long long)T, a64 + S);
}

// Sums of split j (of rs) of sequence q over 32 experts.  rs == 1: final
// P and counts; rs > 1: partial sums part_P / part_c [n_seq, rs, E].
__global__ void __launch_bounds__(1024)
    balance_seq_kernel(const float* __restrict__ sp,
                       const uint8_t* __restrict__ flags, int T, int E, int S,
                       int rs, float* __restrict__ P,
                       int32_t* __restrict__ counts,
                       float* __restrict__ part_P,
                       int32_t* __restrict__ part_c) {
  __shared__ float ps[32][33];
  __shared__ int pc[32][33];
  const int c = threadIdx.x & 31, r = threadIdx.x >> 5;
  const int q = blockIdx.x, e = blockIdx.y * 32 + c, j = blockIdx.z;
  int a, b;
  seq_range(q, S, T, a, b);
  const int Ts = b - a, chunk = (Ts + rs - 1) / rs;
  const int c0 = min(Ts, j * chunk), c1 = min(Ts, c0 + chunk);
  const int n = c1 - c0, per = (n + 31) / 32;
  const int t0 = a + c0 + min(n, r * per), t1 = a + c0 + min(n, (r + 1) * per);
  float sum = 0.f;
  int cnt = 0;
  if (e < E) {
#pragma unroll 4
    for (int t = t0; t < t1; ++t) {
      sum = __fadd_rn(sum, sp[(size_t)t * E + e]);
      cnt += flags[(size_t)t * E + e];
    }
  }
  ps[r][c] = sum;
  pc[r][c] = cnt;
  __syncthreads();
  if (r != 0 || e >= E) return;
  float tot = 0.f;
  int nt = 0;
  for (int i = 0; i < 32; ++i) {
    tot = __fadd_rn(tot, ps[i][c]);
    nt += pc[i][c];
  }
  if (rs == 1) {
    P[(size_t)q * E + e] = __fdiv_rn(tot, (float)Ts);
    counts[(size_t)q * E + e] = nt;
  } else {
    const size_t o = ((size_t)q * rs + j) * E + e;
    part_P[o] = tot;
    part_c[o] = nt;
  }
}

__global__ void __launch_bounds__(1024)
    balance_loss_kernel(float* __restrict__ P, int32_t* __restrict__ counts,
                        const float* __restrict__ part_P,
                        const int32_t* __restrict__ part_c, int rs, int T,
                        int E, int K, int S, float alpha,
                        float* __restrict__ loss) {
  __shared__ float wsum[32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5, q = blockIdx.x;
  int a, b;
  seq_range(q, S, T, a, b);
  float term = 0.f;
  if (e < E) {
    const size_t o = (size_t)q * E + e;
    float Pe;
    int ce;
    if (rs == 1) {
      Pe = P[o];
      ce = counts[o];
    } else {
      float tot = 0.f;
      ce = 0;
#pragma unroll 8
      for (int j = 0; j < rs; ++j) {
        const size_t po = ((size_t)q * rs + j) * E + e;
        tot = __fadd_rn(tot, part_P[po]);
        ce += part_c[po];
      }
      Pe = __fdiv_rn(tot, (float)(b - a));
      P[o] = Pe;
      counts[o] = ce;
    }
    const float f = __fdiv_rn(__fmul_rn((float)E, (float)ce),
                              (float)(K * (b - a)));
    term = __fmul_rn(f, Pe);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    term = __fadd_rn(term, __shfl_xor_sync(0xffffffffu, term, off));
  if (lane == 0) wsum[warp] = term;
  __syncthreads();
  if (e != 0) return;
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot = __fadd_rn(tot, wsum[w]);
  loss[q] = __fmul_rn(alpha, tot);
}

// ===================================================================
// Backward of routing to the router logits (training side of §1.4).  The
// top-K choices and the balance loss's indicator counts are piecewise
// constant in z and carry no gradient; the bias takes no part.  One warp
// per token; s is the forward's sigmoid.
//   gates:    g_k = s_k / D, D = sum of the chosen s;
//             dz_m = s_m (1 - s_m) / D * (dgate_m - sum_k dgate_k g_k)
//             for a chosen m, 0 for the rest
//   balance:  dz_i = dloss_q alpha / T_s * s_i (1 - s_i) / S
//                    * (f_i - sum_j f_j s_j / S),  S = sum_j s_j
// With `accumulate` the row is added to dz, else it overwrites it.
// ===================================================================
template <int EPL, int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
    route_backward_kernel(const float* __restrict__ logits,
                          const int32_t* __restrict__ idx,
                          const float* __restrict__ dgate, int T, int E,
                          int K, int accumulate, float* __restrict__ dz,
                          DevStatus* st) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * WARPS + warp;
  if (t >= T) return;
  const bool active = lane < E / EPL;
  int e = -1;
  float s = 0.f, dg = 0.f;
  if (lane < K) {
    e = idx[(size_t)t * K + lane];
    if (e >= 0 && e < E) {
      s = sigmoid_f32(logits[(size_t)t * E + e]);
      dg = dgate[(size_t)t * K + lane];
    } else {
      record_error(st, MOE_ERR_DEVICE_BOUNDS, 50);
      e = -1;
    }
  }
  float D = s;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    D = __fadd_rn(D, __shfl_xor_sync(0xffffffffu, D, off));
  const float rD = D > 0.f ? __frcp_rn(D) : 0.f;
  float dot = __fmul_rn(dg, __fmul_rn(s, rD));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    dot = __fadd_rn(dot, __shfl_xor_sync(0xffffffffu, dot, off));
  const float c = __fmul_rn(__fmul_rn(__fmul_rn(s, __fsub_rn(1.f, s)), rD),
                            __fsub_rn(dg, dot));
  float o[EPL];
  if (active && accumulate) {
    load_row<EPL>(dz + (size_t)t * E + lane * EPL, o);
  } else {
#pragma unroll
    for (int j = 0; j < EPL; ++j) o[j] = 0.f;
  }
  for (int k = 0; k < K; ++k) {
    const int ek = __shfl_sync(0xffffffffu, e, k);
    const float ck = __shfl_sync(0xffffffffu, c, k);
    if (ek >= 0 && lane == ek / EPL) {
      const int jj = ek - lane * EPL;
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (j == jj) o[j] = __fadd_rn(o[j], ck);
    }
  }
  if (active) store_row<EPL>(dz + (size_t)t * E + lane * EPL, o);
}

template <int EPL, int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
    balance_backward_kernel(const float* __restrict__ logits, int T, int E,
                            int K, int S, float alpha,
                            const int32_t* __restrict__ counts,
                            const float* __restrict__ dloss, int accumulate,
                            float* __restrict__ dz) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * WARPS + warp;
  if (t >= T) return;
  const bool active = lane < E / EPL;
  const int q = t / S;
  int a, b;
  seq_range(q, S, T, a, b);
  const int Ts = b - a;
  float s[EPL], f[EPL];
  if (active) {
    load_row<EPL>(logits + (size_t)t * E + lane * EPL, s);
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      s[j] = sigmoid_f32(s[j]);
      f[j] = __fdiv_rn(
          __fmul_rn((float)E,
                    (float)counts[(size_t)q * E + lane * EPL + j]),
          (float)(K * Ts));
    }
  } else {
#pragma unroll
    for (int j = 0; j < EPL; ++j) s[j] = f[j] = 0.f;
  }
  float Ssum = 0.f, dot = 0.f;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    Ssum = __fadd_rn(Ssum, s[j]);
    dot = __fadd_rn(dot, __fmul_rn(f[j], s[j]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Ssum = __fadd_rn(Ssum, __shfl_xor_sync(0xffffffffu, Ssum, off));
    dot = __fadd_rn(dot, __shfl_xor_sync(0xffffffffu, dot, off));
  }
  const float rS = __frcp_rn(Ssum);
  dot = __fmul_rn(dot, rS);
  const float pre = __fdiv_rn(
      __fmul_rn(dloss != nullptr ? dloss[q] : 1.f, alpha), (float)Ts);
  if (!active) return;
  float o[EPL];
  if (accumulate) load_row<EPL>(dz + (size_t)t * E + lane * EPL, o);
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const float gj = __fmul_rn(
        __fmul_rn(__fmul_rn(pre, __fmul_rn(s[j], __fsub_rn(1.f, s[j]))),
                  rS),
        __fsub_rn(f[j], dot));
    o[j] = accumulate ? __fadd_rn(o[j], gj) : gj;
  }
  store_row<EPL>(dz + (size_t)t * E + lane * EPL, o);
}

// Both gradients of one token in one pass (the gates' and the balance
// loss's): the logits row is read once, the sigmoid of every expert is
// taken once, and dz is written once.  The arithmetic and its order are
// those of route_backward_kernel followed by balance_backward_kernel with
// accumulate set (the gates' term is added first, then the balance term),
// so the result equals the two calls' bit for bit.
// (latency-bound: with at most eight experts per lane, eight blocks per SM
// keep the most tokens in flight; wider rows would spill at that register
// budget)
template <int EPL, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, EPL <= 8 ? 8 : 1)
    route_balance_backward_kernel(
        const float* __restrict__ logits, const int32_t* __restrict__ idx,
        const float* __restrict__ dgate, int T, int E, int K, int S,
        float alpha, const int32_t* __restrict__ counts,
        const float* __restrict__ dloss, int accumulate,
        float* __restrict__ dz, DevStatus* st) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * WARPS + warp;
  if (t >= T) return;
  const bool active = lane < E / EPL;
  // ---- the gates' term (lanes k < K hold the k-th chosen expert)
  int e = -1;
  float sk = 0.f, dg = 0.f;
  if (lane < K) {
    e = idx[(size_t)t * K + lane];
    if (e >= 0 && e < E) {
      sk = sigmoid_f32(logits[(size_t)t * E + e]);
      dg = dgate[(size_t)t * K + lane];
    } else {
      record_error(st, MOE_ERR_DEVICE_BOUNDS, 50);
      e = -1;
    }
  }
  float D = sk;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    D = __fadd_rn(D, __shfl_xor_sync(0xffffffffu, D, off));
  const float rD = D > 0.f ? __frcp_rn(D) : 0.f;
  float gdot = __fmul_rn(dg, __fmul_rn(sk, rD));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    gdot = __fadd_rn(gdot, __shfl_xor_sync(0xffffffffu, gdot, off));
  const float c = __fmul_rn(__fmul_rn(__fmul_rn(sk, __fsub_rn(1.f, sk)), rD),
                            __fsub_rn(dg, gdot));
  // ---- the balance term's per-token sums
  const int q = t / S;
  int a, b;
  seq_range(q, S, T, a, b);
  const int Ts = b - a;
  float s[EPL], f[EPL];
  if (active) {
    load_row<EPL>(logits + (size_t)t * E + lane * EPL, s);
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      s[j] = sigmoid_f32(s[j]);
      f[j] = __fdiv_rn(
          __fmul_rn((float)E,
                    (float)counts[(size_t)q * E + lane * EPL + j]),
          (float)(K * Ts));
    }
  } else {
#pragma unroll
    for (int j = 0; j < EPL; ++j) s[j] = f[j] = 0.f;
  }
  float Ssum = 0.f, dot = 0.f;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    Ssum = __fadd_rn(Ssum, s[j]);
    dot = __fadd_rn(dot, __fmul_rn(f[j], s[j]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Ssum = __fadd_rn(Ssum, __shfl_xor_sync(0xffffffffu, Ssum, off));
    dot = __fadd_rn(dot, __shfl_xor_sync(0xffffffffu, dot, off));
  }
  const float rS = __frcp_rn(Ssum);
  dot = __fmul_rn(dot, rS);
  const float pre = __fdiv_rn(
      __fmul_rn(dloss != nullptr ? dloss[q] : 1.f, alpha), (float)Ts);
  // ---- dz = (dz or 0) + the gates' term + the balance term
  float o[EPL];
  if (active && accumulate) {
    load_row<EPL>(dz + (size_t)t * E + lane * EPL, o);
  } else {
#pragma unroll
    for (int j = 0; j < EPL; ++j) o[j] = 0.f;
  }
  for (int k = 0; k < K; ++k) {
    const int ek = __shfl_sync(0xffffffffu, e, k);
    const float ck = __shfl_sync(0xffffffffu, c, k);
    if (ek >= 0 && lane == ek / EPL) {
      const int jj = ek - lane * EPL;
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (j == jj) o[j] = __fadd_rn(o[j], ck);
    }
  }
  if (!active) return;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const float gj = __fmul_rn(
        __fmul_rn(__fmul_rn(pre, __fmul_rn(s[j], __fsub_rn(1.f, s[j]))),
                  rS),
        __fsub_rn(f[j], dot));
    o[j] = __fadd_rn(o[j], gj);
  }
  store_row<EPL>(dz + (size_t)t * E + lane * EPL, o);
}

// histogram of an existing topk_idx over the same token blocks
__global__ void __launch_bounds__(256)
    block_counts_kernel(const int32_t* __restrict__ topk_idx, int T, int E,
                        int K, int32_t* __restrict__ block_counts,
                        DevStatus* st) {
  __shared__ int cnt[1024];
  for (int i = threadIdx.x; i < E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int t0 = route_block_start(blockIdx.x, T, gridDim.x);
  const int t1 = route_block_start(blockIdx.x + 1, T, gridDim.x);
  for (int p = t0 * K + threadIdx.x; p < t1 * K; p += blockDim.x) {
    const int e = topk_idx[p];
    if (e >= 0 && e < E)
      atomicAdd(&cnt[e], 1);
    else
      record_error(st, MOE_ERR_DEVICE_BOUNDS, 10);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    block_counts[(size_t)blockIdx.x * E + i] = cnt[i];
}

// ===================================================================
// Column scan of the per-block histograms block_counts[nblk][E]: one CTA
// per 32 experts, 1024 threads = 32 expert columns x 32 chunks of block
// rows (a warp reads 32 consecutive counts of one row).
//   counts[e]          = sum over blocks
//   block_prefix[b][e] = sum over blocks b' < b (NULL: not written)
//   bias step on the final counts (bias NULL: none), so a fused forward
//   needs no extra launch.
// ===================================================================
constexpr int kScanCols = 32;

__global__ void __launch_bounds__(1024)
    scan_kernel(const int32_t* __restrict__ block_counts, int nblk, int T,
                int E, int K, int32_t* __restrict__ counts,
                int32_t* __restrict__ block_prefix, float* __restrict__ bias,
                float gamma) {
  __shared__ int part[32][kScanCols + 1];
  const int c = threadIdx.x & 31, r = threadIdx.x >> 5;
  const int e = blockIdx.x * kScanCols + c;
  const bool ve = e < E;
  const int per = (nblk + 31) / 32;
  const int b0 = min(nblk, r * per), b1 = min(nblk, b0 + per);
  int sum = 0;
  if (ve) {
#pragma unroll 8
    for (int b = b0; b < b1; ++b) sum += block_counts[(size_t)b * E + e];
  }
  part[r][c] = sum;
  __syncthreads();
  int pre = 0, tot = 0;
  for (int i = 0; i < 32; ++i) {
    const int v = part[i][c];
    pre += (i < r) ? v : 0;
    tot += v;
  }
  if (!ve) return;
  if (block_prefix != nullptr) {
    int run = pre;
    for (int b = b0; b < b1; ++b) {
      block_prefix[(size_t)b * E + e] = run;
      run += block_counts[(size_t)b * E + e];
    }
  }
  if (r == 0) {
    if (counts != nullptr) counts[e] = tot;
    if (bias != nullptr) {
      const long long lhs = (long long)tot * E, rhs = (long long)T * K;
      const float bv = bias[e];
      bias[e] = lhs > rhs ? __fsub_rn(bv, gamma)
                          : (lhs < rhs ? __fadd_rn(bv, gamma) : bv);
    }
  }
}

// ===================================================================
// Bias step and load statistics from a count vector (one CTA):
//   b_e -= gamma if c_e*E > T*K, += gamma if below, unchanged at the mean;
//   load_stats = {max c, T*K/E, min c}.
// ===================================================================
__global__ void __launch_bounds__(1024)
    bias_stats_kernel(const int32_t* __restrict__ counts, int T, int E, int K,
                      float* __restrict__ bias, float gamma,
                      float* __restrict__ load_stats) {
  __shared__ int red_max[32], red_min[32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  const int c = (e < E) ? counts[e] : 0;
  if (bias != nullptr && e < E) {
    const long long lhs = (long long)c * E, rhs = (long long)T * K;
    const float bv = bias[e];
    bias[e] = lhs > rhs ? __fsub_rn(bv, gamma)
                        : (lhs < rhs ? __fadd_rn(bv, gamma) : bv);
  }
  if (load_stats == nullptr) return;
  int mx = (e < E) ? c : INT_MIN, mn = (e < E) ? c : INT_MAX;
  mx = __reduce_max_sync(0xffffffffu, mx);
  mn = __reduce_min_sync(0xffffffffu, mn);
  if (lane == 0) {
    red_max[warp] = mx;
    red_min[warp] = mn;
  }
  __syncthreads();
  if (e == 0) {
    const int nw = (blockDim.x + 31) / 32;
    for (int w = 1; w < nw; ++w) {
      mx = max(mx, red_max[w]);
      mn = min(mn, red_min[w]);
    }
    load_stats[0] = (float)mx;
    load_stats[1] = (float)((double)T * K / E);
    load_stats[2] = (float)mn;
  }
}

// ===================================================================
// Stable dispatch order.  Block = one routing block (at most
// kRouteTokensPerBlock tokens), one warp per 32-token chunk, lane = token.
// Every block first derives the expert
// offsets (exclusive scan of counts over experts); the block's base row
// for expert e is offsets[e] + block_prefix[blk][e].  mask[w][e] has bit l
// set when lane l's token chose e; a token's rank among the block's tokens
// choosing e is (earlier warps' popcounts) + popc(mask & lanes below).
// Block 0 also writes offsets[E+1] and the load statistics.
// ===================================================================
constexpr int kDestWarps = kRouteTokensPerBlock / 32;

__global__ void __launch_bounds__(kDestWarps * 32)
    dest_kernel(const int32_t* __restrict__ topk_idx,
                const int32_t* __restrict__ counts,
                const int32_t* __restrict__ block_prefix, int T, int E, int K,
                int32_t* __restrict__ offsets, int32_t* __restrict__ dest,
                int32_t* __restrict__ src_row,
                float* __restrict__ load_stats, DevStatus* st) {
  extern __shared__ uint32_t dsm[];
  uint32_t* mask = dsm;                      // [kDestWarps][E]
  uint32_t* pre = dsm + kDestWarps * E;      // [kDestWarps][E]
  int* offs = reinterpret_cast<int*>(dsm + 2 * kDestWarps * E);  // [E+1]
  __shared__ int wsum[kDestWarps], wmax[kDestWarps], wmin[kDestWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < kDestWarps * E; i += blockDim.x) mask[i] = 0;
  // ---- offsets: exclusive scan of counts over experts, chunk per thread
  {
    const int per = (E + (int)blockDim.x - 1) / (int)blockDim.x;
    const int e_lo = min(E, tid * per), e_hi = min(E, e_lo + per);
    int loc = 0, mx = INT_MIN, mn = INT_MAX;
    for (int e = e_lo; e < e_hi; ++e) {
      const int c = counts[e];
      loc += c;
      mx = max(mx, c);
      mn = min(mn, c);
    }
    int incl = loc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    mn = __reduce_min_sync(0xffffffffu, mn);
    if (lane == 31) wsum[warp] = incl;
    if (lane == 0) {
      wmax[warp] = mx;
      wmin[warp] = mn;
    }
    __syncthreads();
    int run = incl - loc, total = 0;
    for (int w = 0; w < kDestWarps; ++w) {
      run += (w < warp) ? wsum[w] : 0;
      total += wsum[w];
      mx = max(mx, wmax[w]);
      mn = min(mn, wmin[w]);
    }
    for (int e = e_lo; e < e_hi; ++e) {
      offs[e] = run;
      run += counts[e];
    }
    if (tid == 0) offs[E] = total;
    if (blockIdx.x == 0 && tid == 0 && load_stats != nullptr) {
      load_stats[0] = (float)mx;
      load_stats[1] = (float)((double)T * K / E);
      load_stats[2] = (float)mn;
    }
  }
  __syncthreads();
  if (blockIdx.x == 0 && offsets != nullptr)
    for (int e = tid; e <= E; e += blockDim.x) offsets[e] = offs[e];
  const int t = route_block_start(blockIdx.x, T, gridDim.x) + warp * 32 +
                lane;
  const bool valid = t < route_block_start(blockIdx.x + 1, T, gridDim.x);
  if (valid)
    for (int k = 0; k < K; ++k) {
      const int e = topk_idx[(size_t)t * K + k];
      if (e >= 0 && e < E) atomicOr(&mask[warp * E + e], 1u << lane);
    }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    uint32_t run = 0;
    for (int w = 0; w < kDestWarps; ++w) {
      pre[w * E + e] = run;
      run += __popc(mask[w * E + e]);
    }
  }
  __syncthreads();
  if (!valid) return;
  const uint32_t below = (1u << lane) - 1u;
  const int32_t* base = block_prefix + (size_t)blockIdx.x * E;
  const int rows = T * K;
  for (int k = 0; k < K; ++k) {
    const int e = topk_idx[(size_t)t * K + k];
    int r = -1;
    if (e >= 0 && e < E)
      r = offs[e] + base[e] + (int)pre[warp * E + e] +
          __popc(mask[warp * E + e] & below);
    if (r >= 0 && r < rows) {
      src_row[r] = t * K + k;
    } else {
      r = -1;
      record_error(st, MOE_ERR_DEVICE_BOUNDS, 11);
    }
    dest[(size_t)t * K + k] = r;
  }
}

// ===================================================================
// Gather (dispatch): xp[dest[t,k]] = x[t].  One block per token reads the
// row once (16-byte vectors) and writes it K times.
// ===================================================================
constexpr int kRowThreads = 128;
constexpr int kMaxVecPerThread = 16;  // H <= 128*16*8 = 16384

__global__ void __launch_bounds__(kRowThreads)
    gather_kernel(const uint16_t* __restrict__ x,
                  const int32_t* __restrict__ dest, int H, int K, int rows,
                  uint16_t* __restrict__ xp) {
  const int t = blockIdx.x;
  const int nvec = H / 8;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  uint4 v[kMaxVecPerThread];
#pragma unroll
  for (int i = 0; i < kMaxVecPerThread; ++i) {
    const int c = threadIdx.x + i * kRowThreads;
    if (c < nvec) v[i] = __ldg(src + c);
  }
  for (int k = 0; k < K; ++k) {
    const int r = __ldg(dest + (size_t)t * K + k);
    if (r < 0 || r >= rows) continue;  // invalid slot: written nowhere
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)r * H);
#pragma unroll
    for (int i = 0; i < kMaxVecPerThread; ++i) {
      const int c = threadIdx.x + i * kRowThreads;
      if (c < nvec) dst[c] = v[i];
    }
  }
}

// ===================================================================
// Combine (eq. 12): out_t = bf16(x_t + ys_t + sum_k g_k * yp[dest[t,k]]),
// fp32 arithmetic, slots in order.  One block per token, 8 bf16 per thread
// per step; for topk <= KU the K expert rows of a step are all requested
// before any is accumulated (the kernel is an HBM stream of 10 rows per
// token), the sum itself still in slot order.  A slot whose dest lies
// outside [0, rows) is skipped: its row is neither loaded nor added (the
// test is uniform across the block, so it costs no divergence).
// ===================================================================
template <int KU>
__global__ void __launch_bounds__(kRowThreads)
    combine_kernel(const uint16_t* __restrict__ x,
                   const uint16_t* __restrict__ ys,
                   const uint16_t* __restrict__ yp,
                   const int32_t* __restrict__ dest,
                   const float* __restrict__ gate, int H, int K, int rows,
                   uint16_t* __restrict__ out) {
  __shared__ int sd[32];
  __shared__ float sg[32];
  const int t = blockIdx.x;
  if (threadIdx.x < K) {
    const int r = dest[(size_t)t * K + threadIdx.x];
    const bool ok = r >= 0 && r < rows;
    sd[threadIdx.x] = ok ? r : -1;
    sg[threadIdx.x] = ok ? gate[(size_t)t * K + threadIdx.x] : 0.f;
  }
  __syncthreads();
  const int nvec = H / 8;
  for (int c = threadIdx.x; c < nvec; c += kRowThreads) {
    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H) + c);
    const uint4 sv =
        __ldg(reinterpret_cast<const uint4*>(ys + (size_t)t * H) + c);
    uint4 yv[KU > 0 ? KU : 1];
    if (KU > 0) {
#pragma unroll
      for (int k = 0; k < KU; ++k)
        if (k < K && sd[k] >= 0)
          yv[k] = __ldg(reinterpret_cast<const uint4*>(yp + (size_t)sd[k] * H) +
                        c);
    }
    const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
    const uint32_t sa[4] = {sv.x, sv.y, sv.z, sv.w};
    float acc[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = bf16_lo(xa[i]) + bf16_lo(sa[i]);
      acc[2 * i + 1] = bf16_hi(xa[i]) + bf16_hi(sa[i]);
    }
    auto add_row = [&](const uint4& v, float g) {
      const uint32_t ya[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(g, bf16_lo(ya[i]), acc[2 * i]);
        acc[2 * i + 1] = fmaf(g, bf16_hi(ya[i]), acc[2 * i + 1]);
      }
    };
    if (KU > 0) {
#pragma unroll
      for (int k = 0; k < KU; ++k)
        if (k < K && sd[k] >= 0) add_row(yv[k], sg[k]);
    } else {
      for (int k = 0; k < K; ++k)
        if (sd[k] >= 0)
          add_row(__ldg(reinterpret_cast<const uint4*>(yp + (size_t)sd[k] * H) +
                        c),
                  sg[k]);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(out + (size_t)t * H)[c] = o;
  }
}
}  // namespace

// ------------------------------------------------------------ launchers
cudaError_t launch_route(const float* logits, const float* bias, int T, int E,
                         int n_group, int topk_group, int topk,
                         int32_t* topk_idx, float* topk_gate,
                         int32_t* block_counts, cudaStream_t s) {
  const int nblk = route_blocks(T);
  const int epl = E <= 32 ? 1 : E / 32;
  const int lpg = (E / n_group) / epl;
  // more warps per block (fewer tokens per warp) while the grid fits on the
  // SMs at once
  const bool wide = nblk <= sm_count() && epl <= 8;
#define MOE_ROUTE_LAUNCH(N, W)                                               \
  {                                                                          \
    const int smem = (W) * RouteWarpSmem<N>::BYTES;                          \
    /* the static histogram (4 KB) counts against the 48 KB default too */  \
    if (cudaFuncSetAttribute(route_kernel<N, W>,                             \
                             cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                             smem) != cudaSuccess)                           \
      return cudaErrorInvalidValue;                                          \
    route_kernel<N, W><<<nblk, (W) * 32, smem, s>>>(                         \
        logits, bias, T, E, n_group, topk_group, topk, lpg, topk_idx,        \
        topk_gate, block_counts);                                            \
  }
#define MOE_ROUTE_CASE(N)                                                    \
  case N:                                                                    \
    if (wide)                                                                \
      MOE_ROUTE_LAUNCH(N, 32)                                                \
    else                                                                     \
      MOE_ROUTE_LAUNCH(N, 16)                                                \
    break;
  // 16 or 32 experts per lane (E = 512, 1024): 16 warps per block only
#define MOE_ROUTE_CASE_NARROW(N)                                             \
  case N:                                                                    \
    MOE_ROUTE_LAUNCH(N, 16)                                                  \
    break;
  switch (epl) {
    MOE_ROUTE_CASE(1)
    MOE_ROUTE_CASE(2)
    MOE_ROUTE_CASE(4)
    MOE_ROUTE_CASE(8)
    MOE_ROUTE_CASE_NARROW(16)
    MOE_ROUTE_CASE_NARROW(32)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_ROUTE_CASE_NARROW
#undef MOE_ROUTE_CASE
#undef MOE_ROUTE_LAUNCH
  return cudaGetLastError();
}

int seq_balance_splits(int T, int E, int seq_len) {
  if (T <= 0 || seq_len <= 0) return 1;
  const long long n_seq = ((long long)T + seq_len - 1) / seq_len;
  const long long base = n_seq * ((E + 31) / 32);
  const long long want = 2LL * kBalSplitTarget;
  if (base >= want) return 1;
  const int smax = (int)std::min<long long>(seq_len, T);
  // at least 256 rows (8 per warp) per split; at most `want` CTAs in all
  // (two 1024-thread CTAs fit an SM: one wave)
  const long long cap = std::max(1, (smax + 255) / 256);
  return (int)std::max<long long>(1, std::min<long long>(want / base, cap));
}

cudaError_t launch_seq_balance(const float* logits, int T, int E, int topk,
                               int seq_len, float alpha, float* sp,
                               uint8_t* flags, float* P, int32_t* counts,
                               float* part_P, int32_t* part_c, float* loss,
                               cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int epl = E <= 32 ? 1 : E / 32;
  const int nblk = (T + kBalTokensPerBlock - 1) / kBalTokensPerBlock;
#define MOE_BAL_CASE(N)                                                   \
  case N:                                                                 \
    balance_token_kernel<N, kBalWarps><<<nblk, kBalWarps * 32, 0, s>>>(   \
        logits, T, E, topk, sp, flags);                                     \
    break;
  switch (epl) {
    MOE_BAL_CASE(1)
    MOE_BAL_CASE(2)
    MOE_BAL_CASE(4)
    MOE_BAL_CASE(8)
    MOE_BAL_CASE(16)
    MOE_BAL_CASE(32)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_BAL_CASE
  const int n_seq = (int)(((long long)T + seq_len - 1) / seq_len);
  const int rs = seq_balance_splits(T, E, seq_len);
  balance_seq_kernel<<<dim3(n_seq, (E + 31) / 32, rs), 1024, 0, s>>>(
      sp, flags, T, E, seq_len, rs, P, counts, part_P, part_c);
  balance_loss_kernel<<<n_seq, ((E + 31) / 32) * 32, 0, s>>>(
      P, counts, part_P, part_c, rs, T, E, topk, seq_len, alpha, loss);
  return cudaGetLastError();
}

cudaError_t launch_route_backward(const float* logits, const int32_t* idx,
                                  const float* dgate, int T, int E, int K,
                                  int accumulate, float* dz, DevStatus* st,
                                  cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int epl = E <= 32 ? 1 : E / 32;
  const int nblk = (T + kBalWarps - 1) / kBalWarps;
#define MOE_RB_CASE(N)                                                      \
  case N:                                                                   \
    route_backward_kernel<N, kBalWarps><<<nblk, kBalWarps * 32, 0, s>>>(    \
        logits, idx, dgate, T, E, K, accumulate, dz, st);                   \
    break;
  switch (epl) {
    MOE_RB_CASE(1)
    MOE_RB_CASE(2)
    MOE_RB_CASE(4)
    MOE_RB_CASE(8)
    MOE_RB_CASE(16)
    MOE_RB_CASE(32)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_RB_CASE
  return cudaGetLastError();
}

cudaError_t launch_seq_balance_backward(const float* logits, int T, int E,
                                        int K, int seq_len, float alpha,
                                        const int32_t* counts_seq,
                                        const float* dloss, int accumulate,
                                        float* dz, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int epl = E <= 32 ? 1 : E / 32;
  const int nblk = (T + kBalWarps - 1) / kBalWarps;
#define MOE_BB_CASE(N)                                                      \
  case N:                                                                   \
    balance_backward_kernel<N, kBalWarps><<<nblk, kBalWarps * 32, 0, s>>>(  \
        logits, T, E, K, seq_len, alpha, counts_seq, dloss, accumulate, dz); \
    break;
  switch (epl) {
    MOE_BB_CASE(1)
    MOE_BB_CASE(2)
    MOE_BB_CASE(4)
    MOE_BB_CASE(8)
    MOE_BB_CASE(16)
    MOE_BB_CASE(32)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_BB_CASE
  return cudaGetLastError();
}

cudaError_t launch_route_balance_backward(
    const float* logits, const int32_t* idx, const float* dgate, int T,
    int E, int K, int seq_len, float alpha, const int32_t* counts_seq,
    const float* dloss, int accumulate, float* dz, DevStatus* st,
    cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int epl = E <= 32 ? 1 : E / 32;
  const int nblk = (T + kBalWarps - 1) / kBalWarps;
#define MOE_RBB_CASE(N)                                                     \
  case N:                                                                   \
    route_balance_backward_kernel<N, kBalWarps>                             \
        <<<nblk, kBalWarps * 32, 0, s>>>(logits, idx, dgate, T, E, K,       \
                                         seq_len, alpha, counts_seq, dloss, \
                                         accumulate, dz, st);               \
    break;
  switch (epl) {
    MOE_RBB_CASE(1)
    MOE_RBB_CASE(2)
    MOE_RBB_CASE(4)
    MOE_RBB_CASE(8)
    MOE_RBB_CASE(16)
    MOE_RBB_CASE(32)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_RBB_CASE
  return cudaGetLastError();
}

cudaError_t launch_block_counts(const int32_t* topk_idx, int T, int E,
                                int topk, int32_t* block_counts,
                                DevStatus* st, cudaStream_t s) {
  block_counts_kernel<<<route_blocks(T), 256, 0, s>>>(topk_idx, T, E, topk,
                                                      block_counts, st);
  return cudaGetLastError();
}

cudaError_t launch_scan(const int32_t* block_counts, int T, int E, int topk,
                        int32_t* counts, int32_t* block_prefix, float* bias,
                        float gamma, cudaStream_t s) {
  const int grid = (E + kScanCols - 1) / kScanCols;
  scan_kernel<<<grid, 1024, 0, s>>>(block_counts, route_blocks(T), T, E,
                                    topk, counts, block_prefix, bias, gamma);
  return cudaGetLastError();
}

cudaError_t launch_dest(const int32_t* topk_idx, const int32_t* counts,
                        const int32_t* block_prefix, int T, int E, int topk,
                        int32_t* offsets, int32_t* dest, int32_t* src_row,
                        float* load_stats, DevStatus* st, cudaStream_t s) {
  const size_t smem = sizeof(uint32_t) * (2 * kDestWarps * E + E + 1);
  dest_kernel<<<route_blocks(T), kDestWarps * 32, smem, s>>>(
      topk_idx, counts, block_prefix, T, E, topk, offsets, dest, src_row,
      load_stats, st);
  return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* dest, int T, int H,
                          int topk, uint16_t* xp, cudaStream_t s) {
  if (H / 8 > kRowThreads * kMaxVecPerThread) return cudaErrorInvalidValue;
  gather_kernel<<<T, kRowThreads, 0, s>>>(x, dest, H, topk, T * topk, xp);
  return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t* x, const uint16_t* ys,
                           const uint16_t* yp, const int32_t* dest,
                           const float* gate, int T, int H, int topk,
                           uint16_t* out, cudaStream_t s) {
  if (topk <= 8)
    combine_kernel<8><<<T, kRowThreads, 0, s>>>(x, ys, yp, dest, gate, H,
                                                topk, T * topk, out);
  else
    combine_kernel<0><<<T, kRowThreads, 0, s>>>(x, ys, yp, dest, gate, H,
                                                topk, T * topk, out);
  return cudaGetLastError();
}

cudaError_t launch_bias_update(const int32_t* counts, float* bias,
                               float* load_stats, int T, int E, int topk,
                               float gamma, cudaStream_t s) {
  const int threads = ((E + 31) / 32) * 32;
  bias_stats_kernel<<<1, threads, 0, s>>>(counts, T, E, topk, bias, gamma,
                                          load_stats);
  return cudaGetLastError();
}

}  // namespace moe
