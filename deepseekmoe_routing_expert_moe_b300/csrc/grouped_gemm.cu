// Grouped BF16 GEMMs of the expert FFNs on the sm_103a tensor cores.
//
// Every routed expert of the DeepSeek-V3 MoE layer is a SwiGLU FFN with
// three matrices ("02 · DeepSeek-V3" (PaperTrace) §1.1); the shared expert
// has the same form and runs on every token (§1.1, §5.1 treats it as a
// ninth, always-chosen expert).  Rows of the dispatched activations are
// grouped by expert (segments [offsets[e], offsets[e+1])), plus one extra
// segment for the shared expert over all T tokens:
//
//   up   (MODE kUp):   h = silu(A W1^T) * (A W3^T)   A = xp rows | x rows
//   down (MODE kDown): y = h W2^T
//
// The same kernel also computes the router logits (MODE kRouter, one
// segment of T token rows): the fp32 router weight is split exactly into
// three bf16 parts, W = W_hi + W_mid + W_lo, and z = x W_hi^T + x W_mid^T +
// x W_lo^T accumulates all three into one fp32 accumulator -- each bf16 x
// bf16 product is exact, so this is an fp32-accumulated x W^T.
//
// Design (one persistent CTA per SM, 6 warps):
//   warp 0 lane 0   TMA producer: A tile 128x64 and B tile BNx64 per stage,
//                   128-byte swizzle, STAGES-deep mbarrier ring
//   warp 1 lane 0   tcgen05.mma issuer (M=128, N=BN, K=16 per instruction),
//                   fp32 accumulators in tensor memory, double buffered;
//                   warp 1 also owns the TMEM allocation
//   warps 2..5      epilogue: tcgen05.ld of the accumulator rows, SwiGLU
//                   (up) or plain conversion (down), bf16 stores of the
//                   rows that belong to the segment
// The work list -- (segment, n-block, m-tile) units, m fastest so that the
// CTAs sharing a weight tile run side by side and hit L2 -- is derived on
// the device from `offsets`; nothing is read back to the host.
//
// Up-projection B tile: rows [0, BN/2) come from W1 and rows [BN/2, BN)
// from W3 for the same BN/2 features, so accumulator column c (gate) pairs
// with column BN/2 + c (up) in the same thread: SwiGLU needs no exchange.
//
// Every wait is bounded (MOE_ERR_TIMEOUT in the status word, then a clean
// exit: in-flight copies and MMAs are drained, TMEM is freed).
#include <cuda.h>

#include <cstdint>
#include <cstring>

#include "device_common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 128;            // tile rows (tokens) = MMA M
constexpr int BK = 64;             // K per stage: 64 bf16 = one 128 B row
constexpr int UMMA_K = 16;         // K of one kind::f16 MMA
constexpr int kThreads = 192;      // 6 warps
constexpr uint64_t kDrainNs = 2000000000ull;


enum { kUp = 0, kDown = 1, kRouter = 2 };
constexpr int kRouterParts = 3;  // W = hi + mid + lo, each bf16
enum {
  kSiteProducer = 21,
  kSiteMmaAcc = 22,
  kSiteMmaFull = 23,
  kSiteEpilogue = 24,
  kSiteDrain = 25,
  kSiteOffsets = 26
};

struct GemmParams {  // CUtensorMap members carry their 64-byte alignment
  CUtensorMap a_routed;   // up: xp [TK, H]      down: h  [TK, I]
  CUtensorMap a_shared;   // up: x  [T, H]       down: hs [T, I_s]
  CUtensorMap b0_routed;  // up: w1 [E*I, H]     down: w2 [E*H, I]
  CUtensorMap b1_routed;  // up: w3 [E*I, H]     down: unused
  CUtensorMap b0_shared;  // up: ws1 [I_s, H]    down: ws2 [H, I_s]
  CUtensorMap b1_shared;  // up: ws3 [I_s, H]    down: unused
  const int32_t* offsets; // [E+1]
  uint16_t* out_routed;   // up: h [TK, I]       down: yp [TK, H]
  uint16_t* out_shared;   // up: hs [T, I_s]     down: ys [T, H]
  DevStatus* status;
  unsigned long long wait_limit_ns;
  int E, T, TK;
  int n_routed, n_shared;  // output columns of a routed / the shared segment
  int k_routed, k_shared;  // reduction length of a routed / the shared one
};

template <int MODE, int BN>
struct Shape {
  static constexpr int OUT_COLS = (MODE == kUp) ? BN / 2 : BN;
  static constexpr int B_PARTS = (MODE == kRouter) ? kRouterParts : 1;
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = B_PARTS * BN * BK * 2;
  static constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulators
  static constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
};

__device__ __forceinline__ void decode_unit(int u, const int* useg,
                                            const int* srows, int NS,
                                            int& s, int& m, int& n) {
  int lo = 0, hi = NS - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (useg[mid] <= u)
      lo = mid;
    else
      hi = mid - 1;
  }
  s = lo;
  const int mt = (srows[s] + BM - 1) / BM;
  const int local = u - useg[s];
  n = local / mt;
  m = local - n * mt;
}

__device__ __forceinline__ float silu_f(float g) {
  return g * __frcp_rn(1.0f + __expf(-g));
}

template <int MODE, int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmParams p) {
  using S = Shape<MODE, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * S::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * S::B_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = bars + 2 * STAGES + 2;
  uint64_t* drain = bars + 2 * STAGES + 4;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(bars + 2 * STAGES + 5);
  // misc[0] TMEM base, misc[1] abort flag, misc[2] bad-offsets flag
  const int E = p.E;
  const int NS = E + 1;  // routed segments + the shared one (index E)
  int* useg = reinterpret_cast<int*>(const_cast<uint32_t*>(misc) + 4);
  int* srows = useg + NS + 1;
  int* srow0 = srows + NS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), 128);
    }
    mbar_init(smem_u32(drain), 1);
    misc[1] = 0;
    misc[2] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.a_routed);
    prefetch_tmap(&p.a_shared);
    prefetch_tmap(&p.b0_routed);
    prefetch_tmap(&p.b0_shared);
    if (MODE == kUp) {
      prefetch_tmap(&p.b1_routed);
      prefetch_tmap(&p.b1_shared);
    }
  }
  if (warp == 2) {
    // segment table: rows, first row, and the exclusive prefix of units
    const int nb_r = p.n_routed / S::OUT_COLS;
    const int nb_s = p.n_shared / S::OUT_COLS;
    const int per = (NS + 31) / 32;
    const int lo = min(NS, lane * per), hi = min(NS, lo + per);
    int mine = 0;
    bool bad = false;
    for (int s = lo; s < hi; ++s) {
      int r0 = 0, rows = p.T;
      if (s < E) {
        r0 = p.offsets[s];
        const int r1 = p.offsets[s + 1];
        if (r0 < 0 || r1 < r0 || r1 > p.TK) {
          bad = true;
          r0 = 0;
          rows = 0;
        } else {
          rows = r1 - r0;
        }
      }
      srows[s] = rows;
      srow0[s] = r0;
      mine += ((rows + BM - 1) / BM) * (s < E ? nb_r : nb_s);
    }
    int incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - mine;
    for (int s = lo; s < hi; ++s) {
      useg[s] = run;
      run += ((srows[s] + BM - 1) / BM) * (s < E ? nb_r : nb_s);
    }
    if (lane == 31) useg[NS] = incl;
    if (__any_sync(0xffffffffu, bad) && lane == 0) misc[2] = 1;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(&misc[0])), S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  int total = useg[NS];
  if (misc[2]) {
    if (threadIdx.x == 0)
      record_error(p.status, MOE_ERR_DEVICE_BOUNDS, kSiteOffsets);
    total = 0;
  }
  const uint64_t limit = p.wait_limit_ns;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer
      uint32_t stage = 0, phase = 0, issued = 0;
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        int s, m, n;
        decode_unit(u, useg, srows, NS, s, m, n);
        const bool sh = (s == E);
        const CUtensorMap* ta = sh ? &p.a_shared : &p.a_routed;
        const CUtensorMap* tb0 = sh ? &p.b0_shared : &p.b0_routed;
        const CUtensorMap* tb1 = sh ? &p.b1_shared : &p.b1_routed;
        const int arow = srow0[s] + m * BM;
        const int brow = (sh ? 0 : s * p.n_routed) + n * S::OUT_COLS;
        const int nkb = (sh ? p.k_shared : p.k_routed) / BK;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1,
                                 abort_flag, limit, p.status,
                                 kSiteProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, S::A_BYTES + S::B_BYTES);
          tma_load_2d_hint(smem_u32(sA + stage * S::A_BYTES), ta, kb * BK,
                           arow, fb, pol_a);
          if (MODE == kUp) {
            tma_load_2d_hint(smem_u32(sB + stage * S::B_BYTES), tb0, kb * BK,
                             brow, fb, pol_w);
            tma_load_2d_hint(
                smem_u32(sB + stage * S::B_BYTES + (BN / 2) * BK * 2), tb1,
                kb * BK, brow, fb, pol_w);
          } else if (MODE == kRouter) {
            // the three bf16 parts of the router weight, one below the other
#pragma unroll
            for (int part = 0; part < kRouterParts; ++part)
              tma_load_2d_hint(
                  smem_u32(sB + stage * S::B_BYTES + part * BN * BK * 2), tb0,
                  kb * BK, part * p.n_shared + brow, fb, pol_a);
          } else {
            tma_load_2d_hint(smem_u32(sB + stage * S::B_BYTES), tb0, kb * BK,
                             brow, fb, pol_w);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      // drain: the last min(issued, STAGES) loads must land before exit
      const uint32_t first = issued > STAGES ? issued - STAGES : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait_bounded(smem_u32(&full[i % STAGES]), (i / STAGES) & 1,
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
        int s, m, n;
        decode_unit(u, useg, srows, NS, s, m, n);
        const int nkb = ((s == E) ? p.k_shared : p.k_routed) / BK;
        const int buf = local & 1;
        const uint32_t ap = (local >> 1) & 1;
        if (!mbar_wait_bounded(smem_u32(&tempty[buf]), ap ^ 1, abort_flag,
                               limit, p.status, kSiteMmaAcc))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * BN;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag,
                                 limit, p.status, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * S::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * S::B_BYTES);
#pragma unroll
          for (int part = 0; part < S::B_PARTS; ++part) {
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
              tc_mma_f16(d, sw128_kmajor_desc(a0 + kk * UMMA_K * 2),
                         sw128_kmajor_desc(b0 + part * BN * BK * 2 +
                                           kk * UMMA_K * 2),
                         S::IDESC, (kb | part | kk) != 0);
            }
          }
          any = true;
          tc_commit(smem_u32(&empty[stage]));
          if (++stage == STAGES) {
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
      int s, m, n;
      decode_unit(u, useg, srows, NS, s, m, n);
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
      const bool sh = (s == E);
      const int row_in_seg = m * BM + r;
      const bool valid = row_in_seg < srows[s];
      uint16_t* out = sh ? p.out_shared : p.out_routed;
      const int ld = sh ? p.n_shared : p.n_routed;
      uint16_t* orow = out + (size_t)(srow0[s] + (valid ? row_in_seg : 0)) * ld +
                       (size_t)n * S::OUT_COLS;
      if (MODE == kUp) {
#pragma unroll 1
        for (int c = 0; c < S::OUT_COLS; c += 16) {
          uint32_t g[16], v[16];
          tmem_ld16(tb + c, g);
          tmem_ld16(tb + S::OUT_COLS + c, v);
          tmem_ld_wait();
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float h0 = silu_f(__uint_as_float(g[2 * i])) *
                             __uint_as_float(v[2 * i]);
            const float h1 = silu_f(__uint_as_float(g[2 * i + 1])) *
                             __uint_as_float(v[2 * i + 1]);
            pk[i] = pack_bf16x2(h0, h1);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      } else if (MODE == kRouter) {
        float* frow = reinterpret_cast<float*>(out) +
                      (size_t)(valid ? row_in_seg : 0) * ld +
                      (size_t)n * S::OUT_COLS;
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          uint32_t v[16];
          tmem_ld16(tb + c, v);
          tmem_ld_wait();
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(frow + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2],
                                  v[4 * i + 3]);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          uint32_t v[16];
          tmem_ld16(tb + c, v);
          tmem_ld_wait();
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]),
                                __uint_as_float(v[2 * i + 1]));
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
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

// ---------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType,
                                  cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                         cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// 2-D bf16 row-major [outer, inner] tensor, box [box_outer, 64], 128 B swizzle
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
              uint32_t box_outer) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int BN, int STAGES>
size_t smem_bytes(int E) {
  using S = Shape<MODE, BN>;
  return 1024 + STAGES * (S::A_BYTES + S::B_BYTES) +
         (2 * STAGES + 5) * sizeof(uint64_t) + 4 * sizeof(uint32_t) +
         sizeof(int) * (3 * (E + 1) + 1);
}

template <int MODE, int BN, int STAGES>
int launch_one(const GemmParams& gp, cudaStream_t s) {
  auto kern = grouped_gemm_kernel<MODE, BN, STAGES>;
  const size_t smem = smem_bytes<MODE, BN, STAGES>(gp.E);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  kern<<<sm_count(), kThreads, smem, s>>>(gp);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

constexpr int kStages = 4;

}  // namespace

int router_tile_n(int E) {
  if (E % 64 == 0) return 64;
  if (E % 32 == 0) return 32;
  if (E % 16 == 0) return 16;
  return 0;
}

int launch_router_logits_tc(const uint16_t* x, const uint16_t* w_split,
                            float* logits, int T, int H, int E,
                            DevStatus* status, uint64_t wait_limit_ns,
                            cudaStream_t s) {
  const int bn = router_tile_n(E);
  if (bn == 0) return MOE_ERR_UNSUPPORTED;
  GemmParams g;
  std::memset(&g, 0, sizeof(g));
  const bool ok = make_map(&g.a_shared, x, H, T, BM) &&
                  make_map(&g.b0_shared, w_split, H,
                           (uint64_t)kRouterParts * E, bn);
  if (!ok) return MOE_ERR_CUDA;
  g.a_routed = g.a_shared;
  g.b0_routed = g.b1_routed = g.b1_shared = g.b0_shared;
  g.offsets = nullptr;  // no routed segments: E = 0 below
  g.out_routed = g.out_shared = reinterpret_cast<uint16_t*>(logits);
  g.status = status;
  g.wait_limit_ns = wait_limit_ns;
  g.E = 0;
  g.T = T;
  g.TK = 0;
  g.n_routed = g.n_shared = E;
  g.k_routed = g.k_shared = H;
  switch (bn) {
    case 64:
      return launch_one<kRouter, 64, kStages>(g, s);
    case 32:
      return launch_one<kRouter, 32, kStages>(g, s);
    default:
      return launch_one<kRouter, 16, kStages>(g, s);
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
      cudaSuccess)
    return 148;
  return n;
}

int launch_expert_ffn(const FfnArgs& a, cudaStream_t s) {
  const int TK = a.T * a.topk;
  // ---- up projection + SwiGLU
  GemmParams up;
  std::memset(&up, 0, sizeof(up));
  const int bf = (a.I % 128 == 0 && a.I_shared % 128 == 0) ? 128 : 64;
  bool ok = make_map(&up.a_routed, a.xp, a.H, TK, BM) &&
            make_map(&up.a_shared, a.x, a.H, a.T, BM) &&
            make_map(&up.b0_routed, a.w1, a.H, (uint64_t)a.E * a.I, bf) &&
            make_map(&up.b1_routed, a.w3, a.H, (uint64_t)a.E * a.I, bf) &&
            make_map(&up.b0_shared, a.ws1, a.H, a.I_shared, bf) &&
            make_map(&up.b1_shared, a.ws3, a.H, a.I_shared, bf);
  if (!ok) return MOE_ERR_CUDA;
  up.offsets = a.offsets;
  up.out_routed = a.h;
  up.out_shared = a.hs;
  up.status = a.status;
  up.wait_limit_ns = a.wait_limit_ns;
  up.E = a.E;
  up.T = a.T;
  up.TK = TK;
  up.n_routed = a.I;
  up.n_shared = a.I_shared;
  up.k_routed = a.H;
  up.k_shared = a.H;
  int rc = (bf == 128) ? launch_one<kUp, 256, kStages>(up, s)
                       : launch_one<kUp, 128, kStages>(up, s);
  if (rc != MOE_OK) return rc;
  if (a.between_event != nullptr)
    cudaEventRecord(static_cast<cudaEvent_t>(a.between_event), s);

  // ---- down projection
  GemmParams dn;
  std::memset(&dn, 0, sizeof(dn));
  const int bn = (a.H % 256 == 0) ? 256 : (a.H % 128 == 0 ? 128 : 64);
  ok = make_map(&dn.a_routed, a.h, a.I, TK, BM) &&
       make_map(&dn.a_shared, a.hs, a.I_shared, a.T, BM) &&
       make_map(&dn.b0_routed, a.w2, a.I, (uint64_t)a.E * a.H, bn) &&
       make_map(&dn.b0_shared, a.ws2, a.I_shared, a.H, bn);
  if (!ok) return MOE_ERR_CUDA;
  dn.b1_routed = dn.b0_routed;
  dn.b1_shared = dn.b0_shared;
  dn.offsets = a.offsets;
  dn.out_routed = a.yp;
  dn.out_shared = a.ys;
  dn.status = a.status;
  dn.wait_limit_ns = a.wait_limit_ns;
  dn.E = a.E;
  dn.T = a.T;
  dn.TK = TK;
  dn.n_routed = a.H;
  dn.n_shared = a.H;
  dn.k_routed = a.I;
  dn.k_shared = a.I_shared;
  switch (bn) {
    case 256:
      return launch_one<kDown, 256, kStages>(dn, s);
    case 128:
      return launch_one<kDown, 128, kStages>(dn, s);
    default:
      return launch_one<kDown, 64, kStages>(dn, s);
  }
}

}  // namespace moe
