// FP8 (E4M3) grouped expert GEMMs with fine-grained scales and promotion
// ("02 · DeepSeek-V3" (PaperTrace) §2, mixed precision; SwiGLU experts of
// §1.1): activations carry one fp32 scale per 1 x 128 tile, weights one per
// 128 x 128 block, and every 128-element slice of the reduction -- exactly
// one scale group of both operands -- is summed by the tensor cores on its
// own and then added, times its two scales, into fp32 registers on the CUDA
// cores (the pages' promotion interval N_C = 128).
//
//   up   (kF8Up):   m = silu(A W1^T) * (A W3^T), quantized again to E4M3
//                   per 1 x 128 tile for the down projection
//   down (kF8Down): y = M W2^T, stored as bf16
//
// Same "swap AB" orientation as the BF16 kernels (grouped_gemm.cu): the
// weights are the MMA's M side (128 rows of one scale block), the tokens
// its N side.  A unit is (segment, 128-feature block, chunk of token rows).
// Two pipeline shapes, chosen per launch from the mean rows per expert:
//   decode  chunks of <= 32 rows, 8 partial-sum buffers, 4 promotion warps
//           (an expert sees a few tokens; the layer streams the weights --
//           the bytes FP8 halves)
//   prefill chunks of <= 128 rows (a segment cut into equal chunks), 2 (up)
//           or 4 (down) partial-sum buffers, 8 promotion warps: two per
//           tensor-memory lane quadrant, each promoting half of the columns
//           (the fp32 running sums of 2 x 64 columns stay in its registers)
//
// One persistent CTA per SM:
//   warp 0 lane 0   producer: per 128-wide k-block one stage holding the
//                   weight tile(s) (128 x 128 B each) and the token tile
//                   (chunk rows x 128 B), 128-byte swizzle, one mbarrier
//   warp 1 lane 0   tcgen05.mma kind::f8f6f4 (E4M3 x E4M3 -> f32), M = 128,
//                   N = rows rounded to 16, K = 32, four per k-block into a
//                   fresh partial-sum buffer in tensor memory
//   warps 2..       promotion and epilogue: per k-block tcgen05.ld of the
//                   partial sums, acc += partial * (s_w * s_t) in fp32,
//                   then SwiGLU + E4M3 re-quantization (up) or bf16 (down),
//                   staged in shared memory for row-contiguous stores
// Every wait is bounded (MOE_ERR_TIMEOUT, then a clean exit).
#include <cuda.h>
#include <cuda_fp8.h>

#include <cstdint>
#include <cstring>

#include "device_common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int F_BM = 128;      // weight rows per accumulator = MMA M
constexpr int F_BK = 128;      // k per stage: 128 E4M3 = one 128 B row
constexpr int F_UMMA_K = 32;   // k of one kind::f8f6f4 MMA
constexpr int F_KBMAX = 64;    // k-blocks per unit (K <= 8192)
constexpr int F_EPI0 = 2;      // first epilogue warp
constexpr uint32_t F_W_BYTES = F_BM * F_BK;  // 16 KB
constexpr uint32_t F_TMEM_COLS = 512;
constexpr size_t F_SMEM_LIMIT = 232448;
constexpr uint64_t F_DRAIN_NS = 2000000000ull;

enum { kF8Up = 0, kF8Down = 1 };

// A pipeline shape: NT token rows per unit at most (MMA N), EW promotion /
// epilogue warps (4: one per tensor-memory lane quadrant; 8: two, each with
// half of the columns), EQUAL: cut a segment into equal chunks (else into
// NT-row chunks and a remainder).  The partial-sum buffers fill the 512
// tensor-memory columns: the MMAs run that many k-blocks ahead of the
// promotion, which carries them (and the weight stream behind them) across
// the epilogue's per-unit work.
template <int NT_, int EW_, bool EQUAL_, int STAGES_UP_, int STAGES_DOWN_>
struct F8Pipe {
  static constexpr int NT = NT_;
  static constexpr int EW = EW_;
  static constexpr bool EQUAL = EQUAL_;
  static constexpr int STAGES_UP = STAGES_UP_;
  static constexpr int STAGES_DOWN = STAGES_DOWN_;
  static constexpr int CW = NT / (EW / 4);   // columns per epilogue warp
  static constexpr int THREADS = 32 * (F_EPI0 + EW);
  static constexpr uint32_t T_BYTES = NT * F_BK;
  static_assert(CW % 16 == 0 && EW % 4 == 0, "shape");
};
using F8Decode = F8Pipe<32, 4, false, 5, 9>;
using F8Prefill = F8Pipe<128, 8, true, 3, 4>;
// mean rows per routed expert from which the prefill shape is used
constexpr int kF8PrefillRows = 64;
enum {
  kF8SiteProducer = 31,
  kF8SiteMma = 32,
  kF8SiteEpi = 33,
  kF8SiteDrain = 34,
  kF8SiteOffsets = 35
};

template <int MODE, class P>
struct F8Shape {
  static constexpr int NACC = MODE == kF8Up ? 2 : 1;
  static constexpr uint32_t STAGE = NACC * F_W_BYTES + P::T_BYTES;
  static constexpr int STAGES = MODE == kF8Up ? P::STAGES_UP : P::STAGES_DOWN;
  static constexpr uint32_t RING = STAGES * STAGE;
  static constexpr int NBUF = (int)F_TMEM_COLS / (NACC * P::NT);
  // output staging: NT rows x 128 features (E4M3 codes or bf16)
  static constexpr uint32_t OUT = MODE == kF8Up ? P::NT * 128 : P::NT * 256;
  static constexpr int BARS = 2 * STAGES + 2 * NBUF + 1;
  static_assert(STAGE % 1024 == 0, "swizzle atoms stay aligned");
  static_assert(NBUF >= 2, "tmem");
};

struct F8Params {  // CUtensorMap members carry their 64-byte alignment
  CUtensorMap tok_routed;  // up: xpq [TK, H]    down: hq [TK, I]
  CUtensorMap tok_shared;  // up: xq [T, H]      down: hsq [T, I_s]
  CUtensorMap wa_routed;   // up: w1 [E*I, H]    down: w2 [E*H, I]
  CUtensorMap wb_routed;   // up: w3 [E*I, H]    down: unused
  CUtensorMap wa_shared;   // up: ws1 [I_s, H]   down: ws2 [H, I_s]
  CUtensorMap wb_shared;   // up: ws3 [I_s, H]   down: unused
  const float* ts_routed;  // token scales [TK, K/128]
  const float* ts_shared;  // [T, K/128]
  const float* sa_routed;  // weight block scales [E*N/128, K/128]
  const float* sb_routed;
  const float* sa_shared;  // [N_s/128, K/128]
  const float* sb_shared;
  const int32_t* offsets;  // [E+1]
  uint8_t* q_routed;       // up: m codes [TK, I]
  float* qs_routed;        // up: m scales [TK, I/128]
  uint8_t* q_shared;       // up: [T, I_s]
  float* qs_shared;        // up: [T, I_s/128]
  uint16_t* y_routed;      // down: yp [TK, H]
  uint16_t* y_shared;      // down: ys [T, H]
  DevStatus* status;
  unsigned long long wait_limit_ns;
  int E, T, TK;
  int n_routed, n_shared;  // output features of a routed / the shared expert
  int k_routed, k_shared;  // reduction length of a routed / the shared one
};

struct F8Unit {
  int seg;   // 0 = shared expert, 1 + e = routed expert e
  int f;     // 128-feature block
  int row0;  // first token row of the chunk
  int rows;  // valid rows (1..32)
  int n;     // MMA N: rows rounded up to 16
};

template <class P>
__device__ __forceinline__ F8Unit f8_decode(int u, const int* useg,
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
  F8Unit x;
  x.seg = lo;
  const int R = srows[lo];
  const int nch = (R + P::NT - 1) / P::NT;
  // chunk length: NT (and a remainder), or R cut into nch equal chunks
  // rounded up to 16 rows
  const int cs = P::EQUAL ? (((R + nch - 1) / nch + 15) & ~15) : P::NT;
  const int local = u - useg[lo];
  x.f = local / nch;
  const int c = local - x.f * nch;
  x.row0 = srow0[lo] + c * cs;
  x.rows = min(cs, R - c * cs);
  x.n = (x.rows + 15) & ~15;
  return x;
}

__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc,
                                          uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor, kind::f8f6f4: D f32, A and B E4M3 (format code
// 0), both K-major, dense, shape M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// named barrier of the EW epilogue warps
template <int EW>
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * EW) : "memory");
}

__device__ __forceinline__ uint32_t e4m3_code(float v, float s) {
  return (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(v, s), __NV_SATFINITE,
                                         __NV_E4M3);
}

template <int MODE, class P>
__global__ void __launch_bounds__(P::THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ F8Params p) {
  using S = F8Shape<MODE, P>;
  constexpr int NACC = S::NACC, STAGES = S::STAGES, NBUF = S::NBUF;
  constexpr int NT = P::NT, EW = P::EW, CW = P::CW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* sout = smem + S::RING;                       // output staging
  float* s_t = reinterpret_cast<float*>(sout + S::OUT);  // [KBMAX][NT]
  float* s_w = s_t + NT * F_KBMAX;                      // [NACC][KBMAX]
  float* s_red = s_w + NACC * F_KBMAX;                  // [4][NT]
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_red + 4 * NT);
  uint64_t* full = bars;
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + NBUF;
  uint64_t* drain = tempty + NBUF;
  volatile uint32_t* misc =
      reinterpret_cast<volatile uint32_t*>(bars + S::BARS);
  // misc[0] TMEM base, [1] abort flag, [2] bad offsets, [3..4] the
  // epilogue warps' failure words of even / odd units (two, so that a warp
  // writing the next unit's never overwrites one the others still read)
  const int E = p.E, NS = E + 1;
  int* useg = reinterpret_cast<int*>(const_cast<uint32_t*>(misc) + 8);
  int* srows = useg + NS + 1;
  int* srow0 = srows + NS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < NBUF; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), 32 * EW);
    }
    mbar_init(smem_u32(drain), 1);
    misc[1] = 0;
    misc[2] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tok_routed);
    prefetch_tmap(&p.tok_shared);
    prefetch_tmap(&p.wa_routed);
    prefetch_tmap(&p.wa_shared);
    if (NACC == 2) {
      prefetch_tmap(&p.wb_routed);
      prefetch_tmap(&p.wb_shared);
    }
  }
  if (warp == 2) {
    // segment table and the exclusive prefix of units per segment
    const int nfb_r = p.n_routed / F_BM, nfb_s = p.n_shared / F_BM;
    const int per = (NS + 31) / 32;
    const int lo = min(NS, lane * per), hi = min(NS, lo + per);
    int mine = 0;
    bool bad = false;
    for (int s = lo; s < hi; ++s) {
      int r0 = 0, rows = p.T;
      if (s > 0) {
        r0 = p.offsets[s - 1];
        const int r1 = p.offsets[s];
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
      mine += ((rows + NT - 1) / NT) * (s > 0 ? nfb_r : nfb_s);
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
      run += ((srows[s] + NT - 1) / NT) * (s > 0 ? nfb_r : nfb_s);
    }
    if (lane == 31) useg[NS] = incl;
    if (__any_sync(0xffffffffu, bad) && lane == 0) misc[2] = 1;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(&misc[0])), F_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  int total = useg[NS];
  if (misc[2]) {
    if (threadIdx.x == 0)
      record_error(p.status, MOE_ERR_DEVICE_BOUNDS, kF8SiteOffsets);
    total = 0;
  }
  const uint64_t limit = p.wait_limit_ns;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer
      uint32_t stage = 0, phase = 0, issued = 0;
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_t = policy_evict_last();
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const F8Unit w = f8_decode<P>(u, useg, srow0, srows, NS);
        const bool sh = (w.seg == 0);
        const CUtensorMap* wa = sh ? &p.wa_shared : &p.wa_routed;
        const CUtensorMap* wb = sh ? &p.wb_shared : &p.wb_routed;
        const CUtensorMap* tok = sh ? &p.tok_shared : &p.tok_routed;
        const int wrow = (sh ? 0 : (w.seg - 1) * p.n_routed) + w.f * F_BM;
        const int nkb = (sh ? p.k_shared : p.k_routed) / F_BK;
        const uint32_t tx = NACC * F_W_BYTES + (uint32_t)w.n * F_BK;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1,
                                 abort_flag, limit, p.status,
                                 kF8SiteProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          uint8_t* st = ring + stage * S::STAGE;
          mbar_arrive_expect_tx(fb, tx);
          tma_load_2d_hint(smem_u32(st), wa, kb * F_BK, wrow, fb, pol_w);
          if (NACC == 2)
            tma_load_2d_hint(smem_u32(st + F_W_BYTES), wb, kb * F_BK, wrow,
                             fb, pol_w);
          // token rows [row0, row0 + n) in boxes of 16 rows
          for (int r16 = 0; r16 < w.n; r16 += 16)
            tma_load_2d_hint(smem_u32(st + NACC * F_W_BYTES + r16 * F_BK),
                             tok, kb * F_BK, w.row0 + r16, fb, pol_t);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      const uint32_t first = issued > STAGES ? issued - STAGES : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait_bounded(smem_u32(&full[i % STAGES]), (i / STAGES) & 1,
                          nullptr, F_DRAIN_NS, p.status, kF8SiteDrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA
      uint32_t stage = 0, phase = 0, kc = 0;
      bool any = false;
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const F8Unit w = f8_decode<P>(u, useg, srow0, srows, NS);
        const int nkb = ((w.seg == 0) ? p.k_shared : p.k_routed) / F_BK;
        const uint32_t idesc = idesc_e4m3_f32(F_BM, w.n);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb, ++kc) {
          const uint32_t b = kc % NBUF;
          if (!mbar_wait_bounded(smem_u32(&tempty[b]),
                                 ((kc / NBUF) & 1) ^ 1, abort_flag, limit,
                                 p.status, kF8SiteMma) ||
              !mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag,
                                 limit, p.status, kF8SiteMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sw = smem_u32(ring + stage * S::STAGE);
          const uint32_t stok = sw + NACC * F_W_BYTES;
#pragma unroll
          for (int a = 0; a < NACC; ++a) {
            const uint32_t d = tmem_base + (b * NACC + a) * NT;
#pragma unroll
            for (int kk = 0; kk < F_BK / F_UMMA_K; ++kk)
              tc_mma_f8(d, sw128_kmajor_desc(sw + a * F_W_BYTES + kk * 32),
                        sw128_kmajor_desc(stok + kk * 32), idesc, kk != 0);
          }
          any = true;
          tc_commit(smem_u32(&empty[stage]));
          tc_commit(smem_u32(&tfull[b]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      if (any) {
        tc_commit(smem_u32(drain));
        mbar_wait_bounded(smem_u32(drain), 0, nullptr, F_DRAIN_NS, p.status,
                          kF8SiteDrain);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------- promotion + epilogue
    const int q = warp & 3;                    // TMEM lane quadrant
    const int r = q * 32 + lane;               // weight row of this thread
    const int et = threadIdx.x - 32 * F_EPI0;  // 0 .. 32 * EW - 1
    const int c0 = ((warp - F_EPI0) >> 2) * CW;  // first column of this warp
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    uint32_t kc = 0;
    int it = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++it) {
      const F8Unit w = f8_decode<P>(u, useg, srow0, srows, NS);
      const bool sh = (w.seg == 0);
      const int K = sh ? p.k_shared : p.k_routed;
      const int nkb = K / F_BK;
      const int nfeat = sh ? p.n_shared : p.n_routed;
      // scales of this unit: tokens [nkb][NT] (0 for rows past the chunk)
      // and the weight block(s) [NACC][nkb]
      {
        const float* ts = sh ? p.ts_shared : p.ts_routed;
        for (int i = et; i < NT * nkb; i += 32 * EW) {
          const int j = i / nkb, kb = i - j * nkb;
          s_t[kb * NT + j] =
              j < w.rows ? ts[(size_t)(w.row0 + j) * nkb + kb] : 0.0f;
        }
        const int wb = (sh ? 0 : (w.seg - 1) * (p.n_routed / F_BM)) + w.f;
        for (int i = et; i < NACC * nkb; i += 32 * EW) {
          const int a = i / nkb, kb = i - a * nkb;
          const float* sc = a == 0 ? (sh ? p.sa_shared : p.sa_routed)
                                   : (sh ? p.sb_shared : p.sb_routed);
          s_w[a * F_KBMAX + kb] = sc[(size_t)wb * nkb + kb];
        }
      }
      epi_sync<EW>();
      float acc[NACC][CW];
#pragma unroll
      for (int a = 0; a < NACC; ++a)
#pragma unroll
        for (int j = 0; j < CW; ++j) acc[a][j] = 0.0f;
      // each warp waits for the partial sums itself (bounded); a wait that
      // runs out ends this warp's k-loop, and the vote after the loop stops
      // every epilogue warp together (no warp is left at a barrier)
      int failed = 0;
      for (int kb = 0; kb < nkb; ++kb, ++kc) {
        const uint32_t b = kc % NBUF;
        int okw = 1;
        if (lane == 0)
          okw = mbar_wait_bounded(smem_u32(&tfull[b]), (kc / NBUF) & 1,
                                  abort_flag, limit, p.status, kF8SiteEpi);
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) {
          failed = 1;
          break;
        }
        tc_fence_after();
        float cw[NACC];
#pragma unroll
        for (int a = 0; a < NACC; ++a) cw[a] = s_w[a * F_KBMAX + kb];
        const float* st = s_t + kb * NT + c0;
        // this warp's CW columns, 16 at a time (columns past the MMA's N
        // hold nothing: they are not loaded and add zero)
#pragma unroll
        for (int c = 0; c < CW / 16; ++c) {
          const bool live = c0 + 16 * c < w.n;
          uint32_t v[NACC][16];
#pragma unroll
          for (int a = 0; a < NACC; ++a) {
            if (live)
              tmem_ld16(tmem_base + lane_off + (b * NACC + a) * NT + c0 +
                            16 * c,
                        v[a]);
          }
          float sv[16];
          if (live) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 f4 =
                  *reinterpret_cast<const float4*>(st + 16 * c + 4 * i);
              sv[4 * i] = f4.x;
              sv[4 * i + 1] = f4.y;
              sv[4 * i + 2] = f4.z;
              sv[4 * i + 3] = f4.w;
            }
          }
          tmem_ld_wait();
          if (live) {
#pragma unroll
            for (int a = 0; a < NACC; ++a)
#pragma unroll
              for (int j = 0; j < 16; ++j)
                acc[a][16 * c + j] = fmaf(__uint_as_float(v[a][j]),
                                          cw[a] * sv[j], acc[a][16 * c + j]);
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&tempty[b]));
      }
      // the unit's vote: did any epilogue warp's wait run out?
      {
        volatile uint32_t* fw = misc + 3 + (it & 1);
        if (et == 0) *fw = 0;
        epi_sync<EW>();
        if (failed && lane == 0) *fw = 1;
        epi_sync<EW>();
        if (*fw) break;
      }
      const bool valid_f = w.f * F_BM + r < nfeat;  // always, by shape
      if (MODE == kF8Up) {
        // m = silu(g) * u per token column (into acc[0]); E4M3 per 1 x 128
        // tile: the tile of token j is column j over the 128 rows of this
        // block, its max over the four lane quadrants' warps
#pragma unroll
        for (int j = 0; j < CW; ++j) {
          const float g = acc[0][j];
          acc[0][j] = g / (1.0f + expf(-g)) * acc[NACC - 1][j];
        }
#pragma unroll
        for (int j = 0; j < CW; ++j) {
          const uint32_t mx = __reduce_max_sync(
              0xffffffffu, __float_as_uint(fabsf(acc[0][j])));
          if (lane == (j & 31)) s_red[q * NT + c0 + j] = __uint_as_float(mx);
        }
        epi_sync<EW>();
        uint8_t* codes = sout;  // [NT tokens][128 features]
#pragma unroll
        for (int j = 0; j < CW; ++j) {
          const int col = c0 + j;
          const float amax = fmaxf(fmaxf(s_red[col], s_red[NT + col]),
                                   fmaxf(s_red[2 * NT + col],
                                         s_red[3 * NT + col]));
          const float sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
          codes[col * 128 + r] = (uint8_t)e4m3_code(acc[0][j], sc);
          if (q == 0 && lane == (j & 31) && col < w.rows && valid_f) {
            float* qs = sh ? p.qs_shared : p.qs_routed;
            qs[(size_t)(w.row0 + col) * (nfeat / 128) + w.f] = sc;
          }
        }
        epi_sync<EW>();
        // NT rows x 128 B: each thread stores 32 B of one row per pass
        for (int i = et; i < NT * 4; i += 32 * EW) {
          const int j = i >> 2, c = (i & 3) * 32;
          if (j < w.rows) {
            uint8_t* dst = (sh ? p.q_shared : p.q_routed) +
                           (size_t)(w.row0 + j) * nfeat + w.f * F_BM + c;
            const uint4* src = reinterpret_cast<const uint4*>(
                codes + j * 128 + c);
            reinterpret_cast<uint4*>(dst)[0] = src[0];
            reinterpret_cast<uint4*>(dst)[1] = src[1];
          }
        }
      } else {
        uint16_t* ys = reinterpret_cast<uint16_t*>(sout);  // [NT][128]
#pragma unroll
        for (int j = 0; j < CW; ++j)
          ys[(c0 + j) * 128 + r] =
              __bfloat16_as_ushort(__float2bfloat16_rn(acc[0][j]));
        epi_sync<EW>();
        // NT rows x 256 B: each thread stores 64 B of one row per pass
        for (int i = et; i < NT * 4; i += 32 * EW) {
          const int j = i >> 2, c = (i & 3) * 32;
          if (j < w.rows) {
            uint16_t* dst = (sh ? p.y_shared : p.y_routed) +
                            (size_t)(w.row0 + j) * nfeat + w.f * F_BM + c;
            const uint4* src =
                reinterpret_cast<const uint4*>(ys + j * 128 + c);
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4)
              reinterpret_cast<uint4*>(dst)[i4] = src[i4];
          }
        }
      }
      epi_sync<EW>();  // staging and scales are reused by the next unit
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, F_TMEM_COLS);
  }
}

template <int MODE, class P>
size_t f8_smem_bytes(int E) {
  using S = F8Shape<MODE, P>;
  return 1024 + S::RING + S::OUT +
         sizeof(float) * (P::NT * F_KBMAX + S::NACC * F_KBMAX + 4 * P::NT) +
         S::BARS * sizeof(uint64_t) + 8 * sizeof(uint32_t) +
         sizeof(int) * (3 * (E + 1) + 1);
}

template <int MODE, class P>
int f8_launch(const F8Params& fp, cudaStream_t s) {
  auto kern = fp8_gemm_kernel<MODE, P>;
  const size_t smem = f8_smem_bytes<MODE, P>(fp.E);
  if (smem > F_SMEM_LIMIT) return MOE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  kern<<<gemm_ctas(), P::THREADS, smem, s>>>(fp);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// the pipeline shape for this launch's mean rows per routed expert
template <int MODE>
int f8_launch_shape(const F8Params& fp, cudaStream_t s) {
  const long long mean_rows = fp.E > 0 ? (long long)fp.TK / fp.E : 0;
  return mean_rows >= kF8PrefillRows ? f8_launch<MODE, F8Prefill>(fp, s)
                                     : f8_launch<MODE, F8Decode>(fp, s);
}

}  // namespace

int fp8_ffn_supported(int H, int I, int I_shared, int E) {
  if (H % 128 || I % 128 || I_shared % 128) return 0;
  if (H / 128 > F_KBMAX || I / 128 > F_KBMAX || I_shared / 128 > F_KBMAX)
    return 0;
  return f8_smem_bytes<kF8Up, F8Decode>(E) <= F_SMEM_LIMIT &&
         f8_smem_bytes<kF8Down, F8Decode>(E) <= F_SMEM_LIMIT &&
         f8_smem_bytes<kF8Up, F8Prefill>(E) <= F_SMEM_LIMIT &&
         f8_smem_bytes<kF8Down, F8Prefill>(E) <= F_SMEM_LIMIT;
}

int launch_expert_ffn_fp8(const FfnFp8Args& a, cudaStream_t s) {
  const int TK = a.T * a.topk;
  F8Params up;
  std::memset(&up, 0, sizeof(up));
  bool ok =
      make_tmap_u8(&up.tok_routed, a.xpq, a.H, TK, 16) &&
      make_tmap_u8(&up.tok_shared, a.xq, a.H, a.T, 16) &&
      make_tmap_u8(&up.wa_routed, a.w1, a.H, (uint64_t)a.E * a.I, F_BM) &&
      make_tmap_u8(&up.wb_routed, a.w3, a.H, (uint64_t)a.E * a.I, F_BM) &&
      make_tmap_u8(&up.wa_shared, a.ws1, a.H, a.I_shared, F_BM) &&
      make_tmap_u8(&up.wb_shared, a.ws3, a.H, a.I_shared, F_BM);
  if (!ok) return MOE_ERR_CUDA;
  up.ts_routed = a.xps;
  up.ts_shared = a.xs;
  up.sa_routed = a.w1s;
  up.sb_routed = a.w3s;
  up.sa_shared = a.ws1s;
  up.sb_shared = a.ws3s;
  up.offsets = a.offsets;
  up.q_routed = a.mq;
  up.qs_routed = a.ms;
  up.q_shared = a.msq;
  up.qs_shared = a.mss;
  up.status = a.status;
  up.wait_limit_ns = a.wait_limit_ns;
  up.E = a.E;
  up.T = a.T;
  up.TK = TK;
  up.n_routed = a.I;
  up.n_shared = a.I_shared;
  up.k_routed = a.H;
  up.k_shared = a.H;
  int rc = f8_launch_shape<kF8Up>(up, s);
  if (rc != MOE_OK) return rc;

  F8Params dn;
  std::memset(&dn, 0, sizeof(dn));
  ok = make_tmap_u8(&dn.tok_routed, a.mq, a.I, TK, 16) &&
       make_tmap_u8(&dn.tok_shared, a.msq, a.I_shared, a.T, 16) &&
       make_tmap_u8(&dn.wa_routed, a.w2, a.I, (uint64_t)a.E * a.H, F_BM) &&
       make_tmap_u8(&dn.wa_shared, a.ws2, a.I_shared, a.H, F_BM);
  if (!ok) return MOE_ERR_CUDA;
  dn.wb_routed = dn.wa_routed;
  dn.wb_shared = dn.wa_shared;
  dn.ts_routed = a.ms;
  dn.ts_shared = a.mss;
  dn.sa_routed = a.w2s;
  dn.sb_routed = a.w2s;
  dn.sa_shared = a.ws2s;
  dn.sb_shared = a.ws2s;
  dn.offsets = a.offsets;
  dn.y_routed = a.yp;
  dn.y_shared = a.ys;
  dn.status = a.status;
  dn.wait_limit_ns = a.wait_limit_ns;
  dn.E = a.E;
  dn.T = a.T;
  dn.TK = TK;
  dn.n_routed = a.H;
  dn.n_shared = a.H;
  dn.k_routed = a.I;
  dn.k_shared = a.I_shared;
  return f8_launch_shape<kF8Down>(dn, s);
}

}  // namespace moe
