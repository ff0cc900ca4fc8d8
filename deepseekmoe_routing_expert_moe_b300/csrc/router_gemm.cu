// Router logits on the sm_103a tensor cores.
//
// The affinity of token t for expert e is the sigmoid of z[t,e] = x_t . w_e
// ("02 · DeepSeek-V3" (PaperTrace) §1.3, eq. 15), with the router weight
// kept in fp32.  The fp32 router weight is split exactly into three bf16
// parts, W = W_hi + W_mid + W_lo, and z = x W_hi^T + x W_mid^T + x W_lo^T
// accumulates all three into one fp32 accumulator -- each bf16 x bf16
// product is exact in fp32, so this is an fp32-accumulated x W^T.  An
// optional per-expert additive term o[e] is added in the epilogue.
//
// Design (one persistent CTA per SM, 6 warps):
//   warp 0 lane 0   TMA producer: x tile 128x64 and the three BNx64 parts of
//                   W per stage, 128-byte swizzle, STAGES-deep mbarrier ring
//   warp 1 lane 0   tcgen05.mma issuer (M=128 tokens, N=BN experts, K=16),
//                   fp32 accumulators in tensor memory, double buffered;
//                   warp 1 also owns the TMEM allocation
//   warps 2..5      epilogue: tcgen05.ld of the accumulator rows, fp32
//                   stores of the valid token rows
// Units are (k range ks, expert block n, token tile m), m fastest.  With
// few token tiles (a decode batch has one) the reduction over H is split
// into ksplit ranges so that every SM gets work: each unit then writes an
// fp32 partial sum, and a second kernel adds the partials in range order
// (deterministic) plus the optional offset.  Every wait is bounded
// (MOE_ERR_TIMEOUT in the status word, then a clean exit).
#include <cuda.h>

#include <cstdint>
#include <algorithm>
#include <cstring>

#include "device_common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 128;        // token rows per tile = MMA M
constexpr int BK = 64;         // K per stage: 64 bf16 = one 128 B row
constexpr int UMMA_K = 16;     // K of one kind::f16 MMA
constexpr int kThreads = 192;  // 6 warps
constexpr int kParts = 3;      // W = hi + mid + lo

constexpr uint64_t kDrainNs = 2000000000ull;

enum {
  kSiteProducer = 41,
  kSiteMmaAcc = 42,
  kSiteMmaFull = 43,
  kSiteEpilogue = 44,
  kSiteDrain = 45
};

struct RouterParams {
  CUtensorMap x_map;  // x [T, H] bf16, box 128 x 64
  CUtensorMap w_map;  // w_split [3*E, H] bf16, box BN x 64
  const float* offset;  // [E] or NULL
  float* logits;      // [T, E]
  float* partial;     // [ksplit, T, E] when ksplit > 1
  int ksplit;
  DevStatus* status;
  unsigned long long wait_limit_ns;
  int T, E, H;
};

template <int BN>
struct RShape {
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = kParts * BN * BK * 2;
  // ring depth: as deep as 227 KB of shared memory allows
  static constexpr int STAGES = BN >= 256 ? 2 : (BN >= 128 ? 3 : 4);
  static constexpr uint32_t TMEM_COLS = (2 * BN < 32) ? 32 : 2 * BN;
  static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    router_gemm_kernel(const __grid_constant__ RouterParams p) {
  using S = RShape<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S::STAGES * S::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + S::STAGES * S::B_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + S::STAGES;
  uint64_t* tfull = bars + 2 * S::STAGES;
  uint64_t* tempty = bars + 2 * S::STAGES + 2;
  uint64_t* drain = bars + 2 * S::STAGES + 4;
  volatile uint32_t* misc =
      reinterpret_cast<volatile uint32_t*>(bars + 2 * S::STAGES + 5);
  // misc[0] TMEM base, misc[1] abort flag
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S::STAGES; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), 128);
    }
    mbar_init(smem_u32(drain), 1);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.x_map);
    prefetch_tmap(&p.w_map);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(&misc[0])), S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  const int mt = (p.T + BM - 1) / BM;
  const int per_split = mt * (p.E / BN);
  const int total = per_split * p.ksplit;
  const int nkb_all = p.H / BK;
  const int kper = (nkb_all + p.ksplit - 1) / p.ksplit;
  const uint64_t limit = p.wait_limit_ns;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer
      uint32_t stage = 0, phase = 0, issued = 0;
      const uint64_t pol = policy_evict_last();
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const int ks = u / per_split, v = u - ks * per_split;
        const int n = v / mt, m = v - n * mt;
        const int kb0 = ks * kper, kb1 = min(nkb_all, kb0 + kper);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1,
                                 abort_flag, limit, p.status,
                                 kSiteProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, S::A_BYTES + S::B_BYTES);
          tma_load_2d_hint(smem_u32(sA + stage * S::A_BYTES), &p.x_map,
                           kb * BK, m * BM, fb, pol);
#pragma unroll
          for (int part = 0; part < kParts; ++part)
            tma_load_2d_hint(
                smem_u32(sB + stage * S::B_BYTES + part * BN * BK * 2),
                &p.w_map, kb * BK, part * p.E + n * BN, fb, pol);
          ++issued;
          if (++stage == S::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      const uint32_t first = issued > S::STAGES ? issued - S::STAGES : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait_bounded(smem_u32(&full[i % S::STAGES]), (i / S::STAGES) & 1,
                          nullptr, kDrainNs, p.status, kSiteDrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA
      uint32_t stage = 0, phase = 0;
      bool any = false;
      int local = 0;
      for (int u = blockIdx.x; u < total; u += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t ap = (local >> 1) & 1;
        if (!mbar_wait_bounded(smem_u32(&tempty[buf]), ap ^ 1, abort_flag,
                               limit, p.status, kSiteMmaAcc))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * BN;
        const int ks = u / per_split;
        const int kb0 = ks * kper, kb1 = min(nkb_all, kb0 + kper);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag,
                                 limit, p.status, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * S::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * S::B_BYTES);
#pragma unroll
          for (int part = 0; part < kParts; ++part) {
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
              tc_mma_f16(d, sw128_kmajor_desc(a0 + kk * UMMA_K * 2),
                         sw128_kmajor_desc(b0 + part * BN * BK * 2 +
                                           kk * UMMA_K * 2),
                         S::IDESC, ((kb - kb0) | part | kk) != 0);
            }
          }
          any = true;
          tc_commit(smem_u32(&empty[stage]));
          if (++stage == S::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&tfull[buf]));
      }
      if (any) {  // every issued MMA completes before TMEM is released
        tc_commit(smem_u32(drain));
        mbar_wait_bounded(smem_u32(drain), 0, nullptr, kDrainNs, p.status,
                          kSiteDrain);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r = q * 32 + lane;
    int local = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++local) {
      const int ks = u / per_split, v = u - ks * per_split;
      const int n = v / mt, m = v - n * mt;
      const int buf = local & 1;
      const uint32_t ap = (local >> 1) & 1;
      int ok = 0;
      if (lane == 0)
        ok = mbar_wait_bounded(smem_u32(&tfull[buf]), ap, abort_flag, limit,
                               p.status, kSiteEpilogue);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(buf * BN);
      const int t = m * BM + r;
      const bool valid = t < p.T;
      const bool split = p.ksplit > 1;
      float* frow = (split ? p.partial + (size_t)ks * p.T * p.E : p.logits) +
                    (size_t)(valid ? t : 0) * p.E + (size_t)n * BN;
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        uint32_t v[16];
        tmem_ld16(tb + c, v);
        tmem_ld_wait();
        if (!split && p.offset != nullptr) {
          const float* o = p.offset + (size_t)n * BN + c;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            v[i] = __float_as_uint(__uint_as_float(v[i]) + __ldg(o + i));
        }
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(frow + c);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2],
                                v[4 * i + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&tempty[buf]));
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

// logits = sum of the ksplit partial sums in range order (+ offset)
__global__ void router_reduce_kernel(const float* __restrict__ partial,
                                     int ksplit, size_t n, int E,
                                     const float* __restrict__ offset,
                                     float* __restrict__ logits) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    float z = partial[i];
    for (int k = 1; k < ksplit; ++k) z = __fadd_rn(z, partial[k * n + i]);
    if (offset != nullptr) z = __fadd_rn(z, offset[i % E]);
    logits[i] = z;
  }
}

template <int BN>
size_t router_smem_bytes() {
  using S = RShape<BN>;
  return 1024 + S::STAGES * (S::A_BYTES + S::B_BYTES) +
         (2 * S::STAGES + 5) * sizeof(uint64_t) + 4 * sizeof(uint32_t);
}

template <int BN>
int launch_router(const RouterParams& rp, cudaStream_t s) {
  auto kern = router_gemm_kernel<BN>;
  const size_t smem = router_smem_bytes<BN>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  kern<<<sm_count(), kThreads, smem, s>>>(rp);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

int router_ksplit(int T, int H, int E) {
  const int bn = router_tile_n(T, E);
  if (bn == 0 || T <= 0) return 1;
  const int units = ((T + BM - 1) / BM) * (E / bn);
  // split only when the plain grid leaves most SMs idle, into as many
  // ranges as keep the units within one wave
  const int sms = 148;
  if (2 * units > sms) return 1;
  const int ks = sms / units;
  const int nkb = H / BK;
  const int max_ks = nkb / 4;  // at least 4 k-blocks per unit
  int k = ks < 1 ? 1 : (ks > max_ks ? (max_ks < 1 ? 1 : max_ks) : ks);
  // ranges of ceil(nkb / k) blocks: take the count that leaves none empty
  const int kper = (nkb + k - 1) / k;
  return (nkb + kper - 1) / kper;
}

// Experts per tile.  Every tile costs the same three MMAs per 16-wide
// k-step whatever its width (up to 256 columns the tensor core's issue, not
// its arithmetic, sets an MMA's time), so wide tiles cut the router's MMA
// count when the token tiles alone fill the SMs (measured on B300 at 4096
// tokens: 111 -> 88 us live); a decode batch keeps 64-wide tiles, split
// over k (54 vs 65 us).
int router_tile_n(int T, int E) {
  if (T >= 1024) {
    if (E % 256 == 0) return 256;
    if (E % 128 == 0) return 128;
  }
  if (E % 64 == 0) return 64;
  if (E % 32 == 0) return 32;
  if (E % 16 == 0) return 16;
  return 0;
}

int launch_router_logits_tc(const uint16_t* x, const uint16_t* w_split,
                            const float* offset, float* logits,
                            float* partial, int T, int H, int E,
                            DevStatus* status, uint64_t wait_limit_ns,
                            cudaStream_t s) {
  const int bn = router_tile_n(T, E);
  if (bn == 0) return MOE_ERR_UNSUPPORTED;
  RouterParams rp;
  std::memset(&rp, 0, sizeof(rp));
  if (!make_tmap_bf16(&rp.x_map, x, H, T, BM) ||
      !make_tmap_bf16(&rp.w_map, w_split, H, (uint64_t)kParts * E, bn))
    return MOE_ERR_CUDA;
  rp.offset = offset;
  rp.logits = logits;
  rp.ksplit = router_ksplit(T, H, E);
  rp.partial = partial;
  if (rp.ksplit > 1 && partial == nullptr) return MOE_ERR_WORKSPACE;
  rp.status = status;
  rp.wait_limit_ns = wait_limit_ns;
  rp.T = T;
  rp.E = E;
  rp.H = H;
  int rc;
  switch (bn) {
    case 256:
      rc = launch_router<256>(rp, s);
      break;
    case 128:
      rc = launch_router<128>(rp, s);
      break;
    case 64:
      rc = launch_router<64>(rp, s);
      break;
    case 32:
      rc = launch_router<32>(rp, s);
      break;
    default:
      rc = launch_router<16>(rp, s);
  }
  if (rc != MOE_OK || rp.ksplit == 1) return rc;
  const size_t n = (size_t)T * E;
  const int blocks = (int)std::min<size_t>((n + 255) / 256, 4 * 148);
  router_reduce_kernel<<<blocks, 256, 0, s>>>(partial, rp.ksplit, n, E,
                                              offset, logits);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
