// Backward of the expert FFNs and the combine on the sm_103a tensor cores
// (the training side of "02 · DeepSeek-V3" (PaperTrace) §1.1 SwiGLU experts
// and §1.3 eq. 12), for a fixed routing.
//
// With a = x_t the token row of a routed slot (t, k), g = g_{t,k} its gate
// and p = W1 a, q = W3 a, m = silu(p) q, y = W2 m (one expert e):
//   dgate[t,k] = <dout_t, y>              = <W2^T dout_t, m>
//   D          = W2^T dout_t              (dgrad of the down projection)
//   dm = g D,  dq = dm silu(p),  dp = dm q silu'(p)
//   da         = W1^T dp + W3^T dq        (dgrad of the up projections)
//   dW1_e += dp a^T,  dW3_e += dq a^T,  dW2_e += (g dout_t) m^T
// and the same for the shared expert over every token with g = 1; the
// token gradient is dx_t = dout_t + da_shared + sum_k da_{t,k}.
//
// Layout: the routed rows are dispatched into segments padded to 16 rows
// (segment e starts at poff[e] = sum_{e'<e} round16(c_e')), the pad rows
// zero, so every reduction over tokens (the weight gradients) runs in whole
// MMA K-steps of 16 rows and never reads another expert's rows.
//
// Kernels (one stream, nothing read back to the host):
//   bwd_pad_kernel       padded offsets, padded dispatch rows, gate per row
//   bwd_gather_kernel    xpp[r] = x_t, dpp[r] = dout_t for the K rows of t
//   bwd_zero_pad_kernel  zero the pad rows (and their gates)
//   dgrad_gemm_kernel<kRecomp>     p, q (fp32) and g m (bf16) recomputed
//   dgrad_gemm_kernel<kDgradDown>  D = dpp W2 per segment; epilogue: dgate
//                                  partials, dp, dq (bf16)
//   dgrad_gemm_kernel<kDgradUp>    dxpp = dp W1 + dq W3 per segment (bf16)
//   wgrad_gemm_kernel              dW1, dW3, dW2 (fp32, optionally added to
//                                  the caller's), K = the segment's rows
//   bwd_finalize_kernel  dx_t and dgate[t, k]
//
// The GEMMs are persistent tcgen05 kernels like the forward ones: one CTA
// per SM, a TMA producer per operand, one MMA-issuing thread, eight
// epilogue warps, fp32 accumulators in tensor memory.  The dgrad GEMMs read the
// weights transposed: their tiles are loaded as MN-major operands (64
// features x 64 reduction rows per TMA box, 128-byte swizzle) and described
// to the MMA as such, so no transposed copy of any weight is made.  The
// weight-gradient GEMM reads both operands MN-major (token rows are its
// reduction dimension).  Every wait is bounded (MOE_ERR_TIMEOUT in the
// status word, then a clean exit).
#include <cuda.h>

#include <cstdint>
#include <cstring>

#include "device_common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 128;       // MMA M
constexpr int BK = 64;        // reduction rows per pipeline stage
constexpr int UMMA_K = 16;    // K of one kind::f16 MMA
constexpr int kPadRows = 16;  // routed segments are padded to this
constexpr int NT = 192;       // largest token chunk (MMA N) of the dgrad GEMMs
constexpr int WSTAGES = 4;    // weight ring depth
constexpr int TSTAGES = 3;    // token ring depth
// eight epilogue warps: two per tensor-memory lane quadrant, each taking
// half of a unit's 16-column chunks (a unit wider than 128 tokens holds
// both accumulator slots, so the MMAs of the next unit wait for its
// epilogue: the shorter the epilogue, the less they wait)
constexpr int kEpiWarps = 8;
constexpr int kEpiWarp0 = 3;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int SLOT = 256;
constexpr int kTokBoxes = 4;
constexpr uint32_t TILE_BYTES = BM * BK * 2;            // 16 KB
constexpr uint32_t WSTAGE_BYTES = 2 * TILE_BYTES;       // two weight tiles
constexpr uint32_t TSTAGE_BYTES = NT * BK * 2;          // 24 KB
constexpr uint32_t TMEM_COLS = 2 * SLOT;
constexpr size_t kSmemLimit = 232448;
constexpr uint64_t kDrainNs = 2000000000ull;
constexpr int kEpiBar = 1;    // named barrier of the dgrad epilogue warps

enum { kRecomp = 0, kDgradDown = 1, kDgradUp = 2 };
enum {
  kSiteProducer = 41,
  kSiteMmaAcc = 42,
  kSiteMmaFull = 43,
  kSiteEpilogue = 44,
  kSiteDrain = 45,
  kSiteOffsets = 46
};

__device__ __forceinline__ int round16(int v) { return (v + 15) & ~15; }

__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync %0, %1;" ::"r"(kEpiBar), "r"(32 * kEpiWarps)
               : "memory");
}

// Shared-memory descriptor of an MN-major operand tile written by TMA with
// 128-byte swizzle in boxes of 64 (M or N) elements x 64 reduction rows:
// each box is 64 rows of 128 B (8-row swizzle atoms, 1024 B apart: the
// stride byte offset), and consecutive 64-element blocks along M / N sit
// 8192 B apart (the leading byte offset).  Fields as in sw128_kmajor_desc.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(8192u >> 4) << 16;  // LBO: next 64-wide block
  d |= static_cast<uint64_t>(1024u >> 4) << 32;  // SBO: next 8 rows of K
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;          // SWIZZLE_128B
  return d;
}

// instruction-descriptor bits: A (bit 15) / B (bit 16) read MN-major
constexpr uint32_t kAMajorMN = 1u << 15;
constexpr uint32_t kBMajorMN = 1u << 16;

// sigma(v) with the exponent's argument capped as in the forward's silu
__device__ __forceinline__ float sigm_f(float v) {
  return __fdividef(1.0f, 1.0f + __expf(fminf(-v, 80.0f)));
}
__device__ __forceinline__ float silu_fwd(float g) {
  return __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f)));
}

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  return static_cast<uint16_t>(pack_bf16x2(v, 0.0f) & 0xFFFFu);
}

// --------------------------------------------------------------------------
// small kernels
// --------------------------------------------------------------------------
// poff[e] = sum_{e'<e} round16(counts[e']) (block scan, every block), block
// 0 writes poff[0..E]; slot i = t*K + k: pdest[i] = dest[i] - off[e] +
// poff[e] (-1 for an invalid slot), gp[pdest[i]] = gate[i]
constexpr int kPadThreads = 256;

__global__ void __launch_bounds__(kPadThreads)
    bwd_pad_kernel(const int32_t* __restrict__ idx,
                   const int32_t* __restrict__ dest,
                   const int32_t* __restrict__ offsets,
                   const int32_t* __restrict__ counts,
                   const float* __restrict__ gate, int TK, int E, int cap,
                   int32_t* __restrict__ poff_out,
                   int32_t* __restrict__ pdest, float* __restrict__ gp,
                   int* __restrict__ ticket, DevStatus* st) {
  __shared__ int poff[1025];
  __shared__ int wsum[kPadThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (E + kPadThreads - 1) / kPadThreads;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int loc = 0;
  for (int e = e0; e < e1; ++e) loc += round16(counts[e]);
  int incl = loc;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int run = incl - loc, total = 0;
  for (int w = 0; w < kPadThreads / 32; ++w) {
    run += (w < warp) ? wsum[w] : 0;
    total += wsum[w];
  }
  for (int e = e0; e < e1; ++e) {
    poff[e] = run;
    run += round16(counts[e]);
  }
  if (tid == 0) poff[E] = total;
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = tid; e <= E; e += kPadThreads) poff_out[e] = poff[e];
    if (tid == 0) *ticket = 0;  // the weight-gradient kernel's task counter
  }
  const int i = blockIdx.x * kPadThreads + tid;
  if (i >= TK) return;
  const int e = idx[i];
  const int r = dest[i];
  int pr = -1;
  if (e >= 0 && e < E && r >= 0) pr = r - offsets[e] + poff[e];
  if (pr < 0 || pr >= cap) {
    pr = -1;
    if (e >= 0 && e < E && r >= 0) record_error(st, MOE_ERR_DEVICE_BOUNDS, 47);
  } else {
    gp[pr] = gate[i];
  }
  pdest[i] = pr;
}

constexpr int kRowThreads = 128;
constexpr int kMaxVec = 16;  // H <= 128 * 16 * 8

// xpp[pdest[t,k]] = x_t, dpp[pdest[t,k]] = dout_t
__global__ void __launch_bounds__(kRowThreads)
    bwd_gather_kernel(const uint16_t* __restrict__ x,
                      const uint16_t* __restrict__ dout,
                      const int32_t* __restrict__ pdest, int H, int K,
                      uint16_t* __restrict__ xpp, uint16_t* __restrict__ dpp) {
  const int t = blockIdx.x;
  const int nvec = H / 8;
  const uint4* sx = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  const uint4* sd = reinterpret_cast<const uint4*>(dout + (size_t)t * H);
  uint4 vx[kMaxVec], vd[kMaxVec];
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const int c = threadIdx.x + i * kRowThreads;
    if (c < nvec) {
      vx[i] = __ldg(sx + c);
      vd[i] = __ldg(sd + c);
    }
  }
  for (int k = 0; k < K; ++k) {
    const int r = __ldg(pdest + (size_t)t * K + k);
    if (r < 0) continue;
    uint4* ox = reinterpret_cast<uint4*>(xpp + (size_t)r * H);
    uint4* od = reinterpret_cast<uint4*>(dpp + (size_t)r * H);
#pragma unroll
    for (int i = 0; i < kMaxVec; ++i) {
      const int c = threadIdx.x + i * kRowThreads;
      if (c < nvec) {
        ox[c] = vx[i];
        od[c] = vd[i];
      }
    }
  }
}

// the pad rows [poff[e] + c_e, poff[e+1]) of both operands, and their gates
__global__ void __launch_bounds__(kRowThreads)
    bwd_zero_pad_kernel(const int32_t* __restrict__ counts,
                        const int32_t* __restrict__ poff, int H,
                        uint16_t* __restrict__ xpp, uint16_t* __restrict__ dpp,
                        float* __restrict__ gp) {
  const int e = blockIdx.x;
  const int r0 = poff[e] + counts[e], r1 = poff[e + 1];
  const int nvec = H / 8;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int r = r0; r < r1; ++r) {
    uint4* ox = reinterpret_cast<uint4*>(xpp + (size_t)r * H);
    uint4* od = reinterpret_cast<uint4*>(dpp + (size_t)r * H);
    for (int c = threadIdx.x; c < nvec; c += kRowThreads) {
      ox[c] = z;
      od[c] = z;
    }
    if (threadIdx.x == 0) gp[r] = 0.0f;
  }
}

// dgate[t,k] = sum over feature blocks of the partials (in order);
// dx_t = bf16(dout_t + dxs_t + sum_k dxpp[pdest[t,k]]), fp32, slot order
__global__ void __launch_bounds__(kRowThreads)
    bwd_finalize_kernel(const uint16_t* __restrict__ dout,
                        const uint16_t* __restrict__ dxs,
                        const uint16_t* __restrict__ dxpp,
                        const int32_t* __restrict__ pdest,
                        const float* __restrict__ dgp, int nfb, int H, int K,
                        uint16_t* __restrict__ dx, float* __restrict__ dgate) {
  __shared__ int sr[32];
  const int t = blockIdx.x;
  if (threadIdx.x < K) {
    const int r = pdest[(size_t)t * K + threadIdx.x];
    sr[threadIdx.x] = r;
    float s = 0.0f;
    if (r >= 0)
      for (int f = 0; f < nfb; ++f) s += dgp[(size_t)r * nfb + f];
    dgate[(size_t)t * K + threadIdx.x] = s;
  }
  __syncthreads();
  const int nvec = H / 8;
  for (int c = threadIdx.x; c < nvec; c += kRowThreads) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(dout + (size_t)t * H) + c);
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(dxs + (size_t)t * H) + c);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
    float acc[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = bf16_lo(av[i]) + bf16_lo(bv[i]);
      acc[2 * i + 1] = bf16_hi(av[i]) + bf16_hi(bv[i]);
    }
    for (int k = 0; k < K; ++k) {
      const int r = sr[k];
      if (r < 0) continue;
      const uint4 y = __ldg(reinterpret_cast<const uint4*>(dxpp + (size_t)r * H) + c);
      const uint32_t yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += bf16_lo(yv[i]);
        acc[2 * i + 1] += bf16_hi(yv[i]);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(dx + (size_t)t * H)[c] = o;
  }
}

// --------------------------------------------------------------------------
// dgrad-style GEMMs: units (segment, feature block, token chunk), two
// accumulators of 128 features each, tokens as the MMA's N side
// --------------------------------------------------------------------------
struct DgParams {  // CUtensorMap members carry their 64-byte alignment
  CUtensorMap tok_r[kTokBoxes];   // B: recomp xpp | ddown dpp | dup dp
  CUtensorMap tok_s[kTokBoxes];   //    recomp x   | ddown dout | dup dps
  CUtensorMap tok2_r[kTokBoxes];  // dup, second half of K: dq
  CUtensorMap tok2_s[kTokBoxes];  //                         dqs
  CUtensorMap wa_r, wb_r;         // A, routed: recomp w1 / w3 (K-major);
                                  // ddown w2 (MN); dup w1 / w3 (MN)
  CUtensorMap wa_s, wb_s;         // A, shared expert
  const int32_t* poff;            // [E+1] padded segment offsets
  const float* gp;                // [TKP] gate of each padded row
  float *p_r, *q_r, *p_s, *q_s;   // [rows, I] fp32: recomp out, ddown in
  uint16_t *hg_r, *hg_s;          // recomp out: g * silu(p) * q (bf16)
  uint16_t *dp_r, *dq_r, *dp_s, *dq_s;  // ddown out (bf16)
  float* dgp;                     // ddown: dgate partials [TKP, nfb]
  uint16_t *out_r, *out_s;        // dup: dxpp [TKP, H], dxs [T, H]
  DevStatus* status;
  unsigned long long wait_limit_ns;
  int E, T, TKP;
  int n_r, n_s;    // output features of a routed / the shared segment
  int k_r, k_s;    // reduction length (dup: the two halves together)
  int wrows_r;     // A rows per routed expert in its tensor map (ddown: H,
                   // dup: I, recomp: I)
  int nfb;
};

template <int MODE>
struct DgFeat {
  static constexpr int FB = (MODE == kRecomp) ? BM : 2 * BM;
};

struct Unit {
  int seg, f, row0, rows, n;
};

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

// One epilogue thread's view of a dgrad-of-down unit: its two feature
// columns fa, fbb (one per accumulator) of the p, q inputs and the dp, dq
// outputs, over the unit's rows.
struct DdTile {
  const float *p, *q;
  uint16_t *dp, *dq;
  const float* gp;  // NULL: the shared expert (g = 1)
  int row0, rows, ld, fa, fbb;
  bool va, vb;
};

// p, q of both columns and the gate, for the 16 token columns of chunk c:
// v[0] p(fa), v[1] q(fa), v[2] p(fbb), v[3] q(fbb), v[4] g
__device__ __forceinline__ void dd_fetch(const DdTile& t, int c,
                                         float (&v)[5][16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int j = 16 * c + i;
    const bool in = j < t.rows;
    const size_t row = (size_t)(t.row0 + (in ? j : 0));
    v[0][i] = (in && t.va) ? t.p[row * t.ld + t.fa] : 0.0f;
    v[1][i] = (in && t.va) ? t.q[row * t.ld + t.fa] : 0.0f;
    v[2][i] = (in && t.vb) ? t.p[row * t.ld + t.fbb] : 0.0f;
    v[3][i] = (in && t.vb) ? t.q[row * t.ld + t.fbb] : 0.0f;
    v[4][i] = t.gp == nullptr ? 1.0f : (in ? t.gp[row] : 0.0f);
  }
}

// chunk c of a dgrad-of-down unit: D from tensor memory, then per token
// column j: dm = g D, dq = dm silu(p), dp = dm q silu'(p) (bf16), and this
// warp's 32-lane sum of D h (h = silu(p) q) into dgs[j]
__device__ __forceinline__ void dd_chunk(const DdTile& t, int c, uint32_t ta,
                                         uint32_t tb, const float (&v)[5][16],
                                         float* dgs, int lane) {
  uint32_t a[16], b[16];
  tmem_ld16(ta + 16 * c, a);
  tmem_ld16(tb + 16 * c, b);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int j = 16 * c + i;
    float part = 0.0f;
    if (j < t.rows) {
      const size_t row = (size_t)(t.row0 + j);
      const float g = v[4][i];
      if (t.va) {
        const float D = __uint_as_float(a[i]);
        const float pv = v[0][i], qv = v[1][i];
        const float sg = sigm_f(pv);
        const float sl = pv * sg;
        part = D * (sl * qv);
        const float dm = g * D;
        t.dq[row * t.ld + t.fa] = bf16_bits(dm * sl);
        t.dp[row * t.ld + t.fa] =
            bf16_bits(dm * qv * (sg * (1.0f + pv * (1.0f - sg))));
      }
      if (t.vb) {
        const float D = __uint_as_float(b[i]);
        const float pv = v[2][i], qv = v[3][i];
        const float sg = sigm_f(pv);
        const float sl = pv * sg;
        part += D * (sl * qv);
        const float dm = g * D;
        t.dq[row * t.ld + t.fbb] = bf16_bits(dm * sl);
        t.dp[row * t.ld + t.fbb] =
            bf16_bits(dm * qv * (sg * (1.0f + pv * (1.0f - sg))));
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
      part += __shfl_xor_sync(0xffffffffu, part, off);
    if (lane == 0) dgs[j] = part;
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    dgrad_gemm_kernel(const __grid_constant__ DgParams p) {
  constexpr int FB = DgFeat<MODE>::FB;
  constexpr bool kAmn = (MODE != kRecomp);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;
  uint8_t* sT = smem + WSTAGES * WSTAGE_BYTES;
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(sT + TSTAGES * TSTAGE_BYTES);
  uint64_t* wfull = bars;
  uint64_t* wempty = wfull + WSTAGES;
  uint64_t* kfull = wempty + WSTAGES;
  uint64_t* kempty = kfull + TSTAGES;
  uint64_t* tfull = kempty + TSTAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  float* dg_s = reinterpret_cast<float*>(drain + 1);      // [4][NT]
  volatile uint32_t* misc =
      reinterpret_cast<volatile uint32_t*>(dg_s + 4 * NT);
  // misc[0] TMEM base, [1] abort, [2] bad offsets, [4 + (unit parity)]
  // the epilogue's go flags (two, so a flag is never rewritten while a
  // warp may still read it)
  const int E = p.E;
  const int NS = E + 1;
  int* useg = reinterpret_cast<int*>(const_cast<uint32_t*>(misc) + 8);
  int* srows = useg + NS + 1;
  int* srow0 = srows + NS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < WSTAGES; ++i) {
      mbar_init(smem_u32(&wfull[i]), 1);
      mbar_init(smem_u32(&wempty[i]), 1);
    }
    for (int i = 0; i < TSTAGES; ++i) {
      mbar_init(smem_u32(&kfull[i]), 1);
      mbar_init(smem_u32(&kempty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), 32 * kEpiWarps);
    }
    mbar_init(smem_u32(drain), 1);
    misc[1] = 0;
    misc[2] = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    const int nfb_r = (p.n_r + FB - 1) / FB;
    const int nfb_s = (p.n_s + FB - 1) / FB;
    const int per = (NS + 31) / 32;
    const int lo = min(NS, lane * per), hi = min(NS, lo + per);
    int mine = 0;
    bool bad = false;
    for (int s = lo; s < hi; ++s) {
      int r0 = 0, rows = p.T;
      if (s > 0) {
        r0 = p.poff[s - 1];
        const int r1 = p.poff[s];
        if (r0 < 0 || r1 < r0 || r1 > p.TKP) {
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
    tmem_alloc(smem_u32(const_cast<uint32_t*>(&misc[0])), TMEM_COLS);
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
      // ------------------------------------------------ weight producer
      uint32_t stage = 0, phase = 0, issued = 0;
      const uint64_t pol = policy_evict_first();
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const Unit w = decode_unit(u, useg, srow0, srows, NS);
        const bool sh = (w.seg == 0);
        const int nkb = (sh ? p.k_s : p.k_r) / BK;
        const int half = nkb / 2;  // dup: W1 for kb < half, W3 after
        const int f0 = w.f * FB;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&wempty[stage]), phase ^ 1,
                                 abort_flag, limit, p.status,
                                 kSiteProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&wfull[stage]);
          uint8_t* st = sW + stage * WSTAGE_BYTES;
          mbar_arrive_expect_tx(fb, WSTAGE_BYTES);
          if (MODE == kRecomp) {
            // K-major 128 x 64 tiles of W1 and W3 (box 64 x 128 rows)
            const int wrow = (sh ? 0 : (w.seg - 1) * p.n_r) + f0;
            tma_load_2d_hint(smem_u32(st), sh ? &p.wa_s : &p.wa_r, kb * BK,
                             wrow, fb, pol);
            tma_load_2d_hint(smem_u32(st + TILE_BYTES),
                             sh ? &p.wb_s : &p.wb_r, kb * BK, wrow, fb, pol);
          } else {
            // MN-major: 256 features (four 64-wide boxes) x 64 rows of K
            const CUtensorMap* m;
            int krow;
            if (MODE == kDgradDown) {
              m = sh ? &p.wa_s : &p.wa_r;
              krow = (sh ? 0 : (w.seg - 1) * p.wrows_r) + kb * BK;
            } else {
              const bool second = kb >= half;
              m = second ? (sh ? &p.wb_s : &p.wb_r) : (sh ? &p.wa_s : &p.wa_r);
              krow = (sh ? 0 : (w.seg - 1) * p.wrows_r) +
                     (second ? kb - half : kb) * BK;
            }
#pragma unroll
            for (int b = 0; b < 4; ++b)
              tma_load_2d_hint(smem_u32(st + b * (TILE_BYTES / 2)), m,
                               f0 + 64 * b, krow, fb, pol);
          }
          ++issued;
          if (++stage == WSTAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      const uint32_t first = issued > WSTAGES ? issued - WSTAGES : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait_bounded(smem_u32(&wfull[i % WSTAGES]), (i / WSTAGES) & 1,
                          nullptr, kDrainNs, p.status, kSiteDrain);
    }
    __syncwarp();
  } else if (warp == 2) {
    if (lane == 0) {
      // ------------------------------------------------- token producer
      uint32_t stage = 0, phase = 0, issued = 0;
      const uint64_t pol = policy_evict_last();
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const Unit w = decode_unit(u, useg, srow0, srows, NS);
        const bool sh = (w.seg == 0);
        const int nkb = (sh ? p.k_s : p.k_r) / BK;
        const int half = nkb / 2;
        const uint32_t tx = (uint32_t)w.n * BK * 2;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&kempty[stage]), phase ^ 1,
                                 abort_flag, limit, p.status,
                                 kSiteProducer)) {
            ok = false;
            break;
          }
          const bool second = (MODE == kDgradUp) && kb >= half;
          const CUtensorMap* tok =
              second ? (sh ? p.tok2_s : p.tok2_r) : (sh ? p.tok_s : p.tok_r);
          const int kc = (second ? kb - half : kb) * BK;
          const uint32_t fb = smem_u32(&kfull[stage]);
          uint8_t* stok = sT + stage * TSTAGE_BYTES;
          mbar_arrive_expect_tx(fb, tx);
          int off = 0;
#pragma unroll
          for (int b = kTokBoxes - 1; b >= 0; --b) {
            if ((w.n >> 4) & (1 << b)) {
              tma_load_2d_hint(smem_u32(stok + off * BK * 2), &tok[b], kc,
                               w.row0 + off, fb, pol);
              off += 16 << b;
            }
          }
          ++issued;
          if (++stage == TSTAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      const uint32_t first = issued > TSTAGES ? issued - TSTAGES : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait_bounded(smem_u32(&kfull[i % TSTAGES]), (i / TSTAGES) & 1,
                          nullptr, kDrainNs, p.status, kSiteDrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA
      uint32_t wstage = 0, wphase = 0, kstage = 0, kphase = 0;
      uint32_t tph = 0;
      int slot = 0;
      bool any = false;
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const Unit w = decode_unit(u, useg, srow0, srows, NS);
        const int nkb = ((w.seg == 0) ? p.k_s : p.k_r) / BK;
        const bool wide = w.n > SLOT / 2;
        const int s1 = wide ? (slot ^ 1) : slot;
        if (!mbar_wait_bounded(smem_u32(&tempty[slot]),
                               ((tph >> slot) & 1) ^ 1, abort_flag, limit,
                               p.status, kSiteMmaAcc))
          break;
        if (wide && !mbar_wait_bounded(smem_u32(&tempty[s1]),
                                       ((tph >> s1) & 1) ^ 1, abort_flag,
                                       limit, p.status, kSiteMmaAcc))
          break;
        tc_fence_after();
        const uint32_t da = tmem_base + slot * SLOT;
        const uint32_t db = wide ? tmem_base + s1 * SLOT : da + SLOT / 2;
        const uint32_t idesc =
            idesc_bf16_f32(BM, w.n) | (kAmn ? kAMajorMN : 0u);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&wfull[wstage]), wphase,
                                 abort_flag, limit, p.status,
                                 kSiteMmaFull) ||
              !mbar_wait_bounded(smem_u32(&kfull[kstage]), kphase,
                                 abort_flag, limit, p.status,
                                 kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t s0 = smem_u32(sW + wstage * WSTAGE_BYTES);
          const uint32_t st = smem_u32(sT + kstage * TSTAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            const uint64_t bdesc = sw128_kmajor_desc(st + kk * UMMA_K * 2);
            const uint32_t acc = (kb | kk) != 0;
            uint64_t adesc_a, adesc_b;
            if (kAmn) {
              adesc_a = sw128_mnmajor_desc(s0 + kk * UMMA_K * 128);
              adesc_b = sw128_mnmajor_desc(s0 + TILE_BYTES + kk * UMMA_K * 128);
            } else {
              adesc_a = sw128_kmajor_desc(s0 + kk * UMMA_K * 2);
              adesc_b = sw128_kmajor_desc(s0 + TILE_BYTES + kk * UMMA_K * 2);
            }
            tc_mma_f16(da, adesc_a, bdesc, idesc, acc);
            tc_mma_f16(db, adesc_b, bdesc, idesc, acc);
          }
          any = true;
          tc_commit(smem_u32(&wempty[wstage]));
          tc_commit(smem_u32(&kempty[kstage]));
          if (++wstage == WSTAGES) {
            wstage = 0;
            wphase ^= 1;
          }
          if (++kstage == TSTAGES) {
            kstage = 0;
            kphase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&tfull[slot]));
        tph ^= 1u << slot;
        if (wide) {
          tc_commit(smem_u32(&tfull[s1]));
          tph ^= 1u << s1;
        } else {
          slot ^= 1;
        }
      }
      if (any) {
        tc_commit(smem_u32(drain));
        mbar_wait_bounded(smem_u32(drain), 0, nullptr, kDrainNs, p.status,
                          kSiteDrain);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- epilogue
    // One thread takes each go / stop decision and the named barrier of
    // the eight epilogue warps shares it, so the warps never part ways at
    // a barrier.
    const int q = warp & 3;
    const int hw = (warp - kEpiWarp0) >> 2;  // which half of the chunks
    const int r = q * 32 + lane;
    const int et = threadIdx.x - 32 * kEpiWarp0;  // 0..255
    uint32_t tph = 0;
    int slot = 0;
    int it = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++it) {
      const Unit w = decode_unit(u, useg, srow0, srows, NS);
      const bool wide = w.n > SLOT / 2;
      const int s1_ = wide ? (slot ^ 1) : slot;
      if (et == 0) {
        int ok = mbar_wait_bounded(smem_u32(&tfull[slot]), (tph >> slot) & 1,
                                   abort_flag, limit, p.status, kSiteEpilogue);
        if (ok && wide)
          ok = mbar_wait_bounded(smem_u32(&tfull[s1_]), (tph >> s1_) & 1,
                                 abort_flag, limit, p.status, kSiteEpilogue);
        misc[4 + (it & 1)] = ok;
      }
      epi_bar();
      if (!misc[4 + (it & 1)]) break;
      tc_fence_after();
      const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
      const uint32_t ta = tmem_base + lane_off + slot * SLOT;
      const uint32_t tb =
          wide ? tmem_base + lane_off + s1_ * SLOT : ta + SLOT / 2;
      const bool sh = (w.seg == 0);
      const int nfeat = sh ? p.n_s : p.n_r;
      const int nch = (w.n + 15) / 16;
      const int c_lo = hw ? (nch + 1) / 2 : 0;
      const int c_hi = hw ? nch : (nch + 1) / 2;
      if (MODE == kRecomp) {
        const int fa = w.f * FB + r;
        const bool vf = fa < nfeat;
        float* po = sh ? p.p_s : p.p_r;
        float* qo = sh ? p.q_s : p.q_r;
        uint16_t* ho = sh ? p.hg_s : p.hg_r;
        for (int c = c_lo; c < c_hi; ++c) {
          uint32_t a[16], b[16];
          tmem_ld16(ta + 16 * c, a);
          tmem_ld16(tb + 16 * c, b);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int j = 16 * c + i;
            if (vf && j < w.rows) {
              const size_t row = (size_t)(w.row0 + j);
              const float pv = __uint_as_float(a[i]);
              const float qv = __uint_as_float(b[i]);
              const float g = sh ? 1.0f : p.gp[row];
              po[row * nfeat + fa] = pv;
              qo[row * nfeat + fa] = qv;
              ho[row * nfeat + fa] = bf16_bits(g * (silu_fwd(pv) * qv));
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&tempty[slot]));
        if (wide) mbar_arrive(smem_u32(&tempty[s1_]));
      } else if (MODE == kDgradDown) {
        const int fa = w.f * FB + r;
        const int fbb = fa + BM;
        const bool va = fa < nfeat, vb = fbb < nfeat;
        const DdTile t{sh ? p.p_s : p.p_r, sh ? p.q_s : p.q_r,
                       sh ? p.dp_s : p.dp_r, sh ? p.dq_s : p.dq_r,
                       sh ? nullptr : p.gp, w.row0, w.rows, nfeat, fa, fbb,
                       va, vb};
        // each warp's chunks: p, q and the gates loaded, then the chunk
        float s0[5][16];
        for (int c = c_lo; c < c_hi; ++c) {
          dd_fetch(t, c, s0);
          dd_chunk(t, c, ta, tb, s0, dg_s + q * NT, lane);
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&tempty[slot]));
        if (wide) mbar_arrive(smem_u32(&tempty[s1_]));
        epi_bar();
        if (!sh) {
          for (int j = et; j < w.rows; j += 32 * kEpiWarps)
            p.dgp[(size_t)(w.row0 + j) * p.nfb + w.f] =
                ((dg_s[j] + dg_s[NT + j]) + dg_s[2 * NT + j]) +
                dg_s[3 * NT + j];
        }
      } else {
        // dgrad of the up projections: two 128-feature blocks of dx rows
        const int fa = w.f * FB + r;
        const int fbb = fa + BM;
        uint16_t* out = sh ? p.out_s : p.out_r;
        const int ld = nfeat;
        for (int c = c_lo; c < c_hi; ++c) {
          uint32_t a[16], b[16];
          tmem_ld16(ta + 16 * c, a);
          tmem_ld16(tb + 16 * c, b);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int j = 16 * c + i;
            if (j < w.rows) {
              const size_t row = (size_t)(w.row0 + j);
              if (fa < ld) out[row * ld + fa] = bf16_bits(__uint_as_float(a[i]));
              if (fbb < ld)
                out[row * ld + fbb] = bf16_bits(__uint_as_float(b[i]));
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&tempty[slot]));
        if (wide) mbar_arrive(smem_u32(&tempty[s1_]));
      }
      tph ^= 1u << slot;
      if (wide)
        tph ^= 1u << s1_;
      else
        slot ^= 1;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

size_t dgrad_smem_bytes(int E) {
  return 1024 + WSTAGES * WSTAGE_BYTES + TSTAGES * TSTAGE_BYTES +
         (2 * WSTAGES + 2 * TSTAGES + 5) * sizeof(uint64_t) +
         4 * NT * sizeof(float) + 8 * sizeof(uint32_t) +
         sizeof(int) * (3 * (E + 1) + 1);
}

template <int MODE>
int launch_dgrad(const DgParams& dp, cudaStream_t s) {
  auto kern = dgrad_gemm_kernel<MODE>;
  const size_t smem = dgrad_smem_bytes(dp.E);
  if (smem > kSmemLimit) return MOE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  kern<<<gemm_ctas(), kThreads, smem, s>>>(dp);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// --------------------------------------------------------------------------
// weight gradients: tasks (matrix, segment, 256-column block, group of
// 128-row blocks); the reduction runs over the segment's token rows.
//
// Per 128 x 256 fp32 output block the MMA reads a 128-column slice of the
// A side (dp, dq or dpp rows) and a 256-column slice of the B side (xpp or
// hg rows) over the segment's rows.  A segment of at most 192 rows keeps
// its B slice in shared memory for a group of up to 16 row blocks, so each
// further block streams only its A slice (a third of the operand bytes);
// longer segments (the shared expert, skewed experts) stream both per
// block.  The tail of a segment is loaded in 16-row boxes, so no rows past
// it are fetched.  CTAs take tasks from a counter in global memory that the
// dispatch kernel of the same call zeroes: a CTA on a slower path through
// the memory system simply takes fewer tasks.
// --------------------------------------------------------------------------
constexpr int WG_N = 256;
constexpr int WG_ASTAGES = 3;   // A ring: 128 columns x 64 rows (16 KB)
constexpr int WG_BSLOTS = 3;    // B ring: 256 columns x 64 rows (32 KB)
constexpr int WG_GROUP = 16;    // row blocks per task while B is resident
constexpr int WG_QN = 8;        // depth of the task queue in shared memory
constexpr int WG_RES_ROWS = WG_BSLOTS * BK;         // 192
constexpr uint32_t WG_A_BYTES = BM * BK * 2;        // 16 KB
constexpr uint32_t WG_B_BYTES = WG_N * BK * 2;      // 32 KB
constexpr uint32_t WG_BOX_BYTES = 64 * BK * 2;      // one 64 x 64 box, 8 KB
constexpr uint32_t WG_BOX16_BYTES = 64 * 16 * 2;    // one 64 x 16 box, 2 KB
// eight epilogue warps: two per tensor-memory lane quadrant, each storing
// half of a block's columns (the fp32 stores are the kernel's long pole)
constexpr int kWgEpiWarps = 8;
constexpr int kWgThreads = 32 * (kEpiWarp0 + kWgEpiWarps);
// fp32 output staging: per epilogue warp two 32 x 32 tiles (4 KB each),
// stored by TMA (or added to the output in L2 when accumulating)
constexpr int WG_OUT_BUFS = 2;
constexpr uint32_t WG_OUT_TILE = 32 * 32 * 4;
constexpr uint32_t WG_OUT_BYTES = kWgEpiWarps * WG_OUT_BUFS * WG_OUT_TILE;
constexpr int kMats = 3;   // dW1, dW3, dW2
constexpr int kWgBars = 2 * WG_ASTAGES + 2 * WG_BSLOTS + 4 + 2 * WG_QN + 1;
enum { kSiteQueue = 48 };

struct WgParams {
  // routed: (dp, xpp) (dq, xpp) (dpp, hg); shared: (dps, x) (dqs, x)
  // (dout, hs); 64-row boxes and 16-row boxes (segment tails)
  CUtensorMap a_r[kMats], b_r[kMats], a_s[kMats], b_s[kMats];
  CUtensorMap a_r16[kMats], b_r16[kMats], a_s16[kMats], b_s16[kMats];
  CUtensorMap o_r[kMats], o_s[kMats];  // outputs as [experts][M][N] fp32
  const int32_t* poff;
  int* ticket;           // task counter, zero at launch
  float* out_r[kMats];   // dW1, dW3 [E, I, H], dW2 [E, H, I]
  float* out_s[kMats];   // dWs1, dWs3 [I_s, H], dWs2 [H, I_s]
  DevStatus* status;
  unsigned long long wait_limit_ns;
  int E, T, TKP, H, I, Is;
  int accumulate;
};

struct WTask {
  int mat, seg, M, N, rows, row0, n0, nt, mb0, mb1;
  bool res;   // B slice resident for the group
};

// M and N of matrix `mat` for a segment (shared: s == 0)
__device__ __forceinline__ void wg_dims(const WgParams& p, int mat, int s,
                                        int& M, int& N) {
  const int If = s == 0 ? p.Is : p.I;
  M = mat < 2 ? If : p.H;
  N = mat < 2 ? p.H : If;
}

// row blocks per task of a segment with `rows` rows (an empty segment's
// blocks are zero-filled, a group at a time)
__device__ __forceinline__ int wg_group(int rows) {
  return rows <= WG_RES_ROWS ? WG_GROUP : 1;
}

__device__ __forceinline__ int wg_tasks(int M, int N, int rows) {
  const int G = wg_group(rows);
  return ((M + BM - 1) / BM + G - 1) / G * ((N + WG_N - 1) / WG_N);
}

// rows and first row of segment s (0: the shared expert over the T tokens;
// s >= 1: routed expert s - 1 between its padded offsets)
__device__ __forceinline__ int wg_rows(const WgParams& p, const int* spoff,
                                       int s) {
  return s == 0 ? p.T : spoff[s] - spoff[s - 1];
}

__device__ __forceinline__ WTask wg_decode(const WgParams& p, int t,
                                           const int* upre, const int* spoff,
                                           int NP) {
  int lo = 0, hi = NP - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (upre[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int NS = p.E + 1;
  WTask x;
  x.mat = lo / NS;
  x.seg = lo - x.mat * NS;
  wg_dims(p, x.mat, x.seg, x.M, x.N);
  x.rows = wg_rows(p, spoff, x.seg);
  x.row0 = x.seg == 0 ? 0 : spoff[x.seg - 1];
  const int G = wg_group(x.rows);
  const int nb = (x.N + WG_N - 1) / WG_N;
  const int local = t - upre[lo];
  const int g = local / nb;
  x.n0 = (local - g * nb) * WG_N;
  x.nt = min(WG_N, x.N - x.n0);
  x.mb0 = g * G;
  x.mb1 = min((x.M + BM - 1) / BM, x.mb0 + G);
  x.res = x.rows > 0 && x.rows <= WG_RES_ROWS;
  return x;
}

// Reduction rows [row, row + min(left, 64)) of `nbox` 64-column boxes
// (columns x0, x0 + 64, ...) into a stage of 64-row boxes `box_bytes`
// apart.  A tail (left < 64) is fetched in 16-row boxes, which land where
// the 64-row box would put those rows (whole 1 KB swizzle atoms).  Returns
// the bytes the copies deliver.
__device__ __forceinline__ uint32_t wg_load_rows(
    uint32_t dst, const CUtensorMap* m64, const CUtensorMap* m16, int x0,
    int nbox, uint32_t box_bytes, int row, int left, uint32_t bar,
    uint64_t pol) {
  if (left >= BK) {
    for (int b = 0; b < nbox; ++b)
      tma_load_2d_hint(dst + b * box_bytes, m64, x0 + 64 * b, row, bar, pol);
    return nbox * WG_BOX_BYTES;
  }
  const int n16 = (left + 15) / 16;
  for (int j = 0; j < n16; ++j)
    for (int b = 0; b < nbox; ++b)
      tma_load_2d_hint(dst + b * box_bytes + j * WG_BOX16_BYTES, m16,
                       x0 + 64 * b, row + 16 * j, bar, pol);
  return n16 * nbox * WG_BOX16_BYTES;
}

// bytes wg_load_rows delivers (the transaction count of the stage)
__device__ __forceinline__ uint32_t wg_rows_bytes(int nbox, int left) {
  return left >= BK ? nbox * WG_BOX_BYTES
                    : ((left + 15) / 16) * nbox * WG_BOX16_BYTES;
}

__global__ void __launch_bounds__(kWgThreads, 1)
    wgrad_gemm_kernel(const __grid_constant__ WgParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = smem;                            // B ring
  uint8_t* sA = sB + WG_BSLOTS * WG_B_BYTES;     // A ring
  uint8_t* sO = sA + WG_ASTAGES * WG_A_BYTES;    // output staging
  uint64_t* bars = reinterpret_cast<uint64_t*>(sO + WG_OUT_BYTES);
  uint64_t* afull = bars;
  uint64_t* aempty = afull + WG_ASTAGES;
  uint64_t* bfull = aempty + WG_ASTAGES;
  uint64_t* bempty = bfull + WG_BSLOTS;
  uint64_t* tfull = bempty + WG_BSLOTS;
  uint64_t* tempty = tfull + 2;
  uint64_t* qfull = tempty + 2;
  uint64_t* qempty = qfull + WG_QN;
  uint64_t* drain = qempty + WG_QN;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(drain + 1);
  volatile int* qv = reinterpret_cast<volatile int*>(misc + 4);
  const int NS = p.E + 1;
  const int NP = kMats * NS;
  int* upre = const_cast<int*>(qv) + WG_QN;
  int* spoff = upre + NP + 1;   // the padded offsets [E + 1]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < WG_ASTAGES; ++i) {
      mbar_init(smem_u32(&afull[i]), 1);
      mbar_init(smem_u32(&aempty[i]), 1);
    }
    for (int i = 0; i < WG_BSLOTS; ++i) {
      mbar_init(smem_u32(&bfull[i]), 1);
      mbar_init(smem_u32(&bempty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), 32 * kWgEpiWarps);
    }
    // a task id is read by the MMA thread and each epilogue warp
    for (int i = 0; i < WG_QN; ++i) {
      mbar_init(smem_u32(&qfull[i]), 1);
      mbar_init(smem_u32(&qempty[i]), 1 + kWgEpiWarps);
    }
    mbar_init(smem_u32(drain), 1);
    misc[1] = 0;
    misc[2] = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    // the segments' offsets (checked), then tasks per (matrix, segment)
    // pair and their prefix
    bool bad = false;
    for (int e = lane; e < NS; e += 32) {
      const int r1 = p.poff[e];
      const int r0 = e > 0 ? p.poff[e - 1] : 0;
      if (r0 < 0 || r1 < r0 || r1 > p.TKP) bad = true;
      spoff[e] = r1;
    }
    bad = __any_sync(0xffffffffu, bad);
    __syncwarp();
    const int per = (NP + 31) / 32;
    const int lo = min(NP, lane * per), hi = min(NP, lo + per);
    int mine = 0;
    for (int i = lo; i < hi; ++i) {
      const int mat = i / NS, s = i - mat * NS;
      int M, N;
      wg_dims(p, mat, s, M, N);
      mine += bad ? 0 : wg_tasks(M, N, wg_rows(p, spoff, s));
    }
    int incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - mine;
    for (int i = lo; i < hi; ++i) {
      upre[i] = run;
      const int mat = i / NS, s = i - mat * NS;
      int M, N;
      wg_dims(p, mat, s, M, N);
      run += bad ? 0 : wg_tasks(M, N, wg_rows(p, spoff, s));
    }
    if (lane == 31) upre[NP] = incl;
    if (bad && lane == 0) misc[2] = 1;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(&misc[0])), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  int total = upre[NP];
  if (misc[2]) {
    if (threadIdx.x == 0)
      record_error(p.status, MOE_ERR_DEVICE_BOUNDS, kSiteOffsets);
    total = 0;
  }
  const uint64_t limit = p.wait_limit_ns;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------- task queue + operand producer
      uint32_t af = 0, bf = 0, qf = 0;
      const uint64_t pol = policy_evict_last();
      bool ok = true;
      // one stage of the A ring (two 64-column boxes) or the B ring
      auto load_a = [&](const CUtensorMap* m64, const CUtensorMap* m16,
                        int m0, int row, int left) {
        const uint32_t s = af % WG_ASTAGES;
        if (!mbar_wait_bounded(smem_u32(&aempty[s]),
                               ((af / WG_ASTAGES) & 1) ^ 1, abort_flag, limit,
                               p.status, kSiteProducer))
          return false;
        const uint32_t fb = smem_u32(&afull[s]);
        mbar_arrive_expect_tx(fb, wg_rows_bytes(2, left));
        wg_load_rows(smem_u32(sA + s * WG_A_BYTES), m64, m16, m0, 2,
                     WG_BOX_BYTES, row, left, fb, pol);
        ++af;
        return true;
      };
      auto load_b = [&](const CUtensorMap* m64, const CUtensorMap* m16,
                        int n0, int nbox, int row, int left) {
        const uint32_t s = bf % WG_BSLOTS;
        if (!mbar_wait_bounded(smem_u32(&bempty[s]),
                               ((bf / WG_BSLOTS) & 1) ^ 1, abort_flag, limit,
                               p.status, kSiteProducer))
          return false;
        const uint32_t fb = smem_u32(&bfull[s]);
        mbar_arrive_expect_tx(fb, wg_rows_bytes(nbox, left));
        wg_load_rows(smem_u32(sB + s * WG_B_BYTES), m64, m16, n0, nbox,
                     WG_BOX_BYTES, row, left, fb, pol);
        ++bf;
        return true;
      };
      while (ok) {
        int t = atomicAdd(p.ticket, 1);
        if (t >= total) t = -1;
        const uint32_t qs = qf % WG_QN;
        if (!mbar_wait_bounded(smem_u32(&qempty[qs]), ((qf / WG_QN) & 1) ^ 1,
                               abort_flag, limit, p.status, kSiteQueue))
          break;
        qv[qs] = t;
        mbar_arrive(smem_u32(&qfull[qs]));
        ++qf;
        if (t < 0) break;
        const WTask w = wg_decode(p, t, upre, spoff, NP);
        if (w.rows == 0) continue;
        const bool sh = w.seg == 0;
        const CUtensorMap* ma = sh ? &p.a_s[w.mat] : &p.a_r[w.mat];
        const CUtensorMap* mb = sh ? &p.b_s[w.mat] : &p.b_r[w.mat];
        const CUtensorMap* ma16 = sh ? &p.a_s16[w.mat] : &p.a_r16[w.mat];
        const CUtensorMap* mb16 = sh ? &p.b_s16[w.mat] : &p.b_r16[w.mat];
        const int nkb = (w.rows + BK - 1) / BK;
        const int nbox = (w.nt + 63) / 64;
        if (w.res)
          for (int kb = 0; kb < nkb && ok; ++kb)
            ok = load_b(mb, mb16, w.n0, nbox, w.row0 + kb * BK,
                        w.rows - kb * BK);
        for (int mblk = w.mb0; mblk < w.mb1 && ok; ++mblk)
          for (int kb = 0; kb < nkb && ok; ++kb) {
            const int row = w.row0 + kb * BK, left = w.rows - kb * BK;
            if (!w.res) ok = load_b(mb, mb16, w.n0, nbox, row, left);
            if (ok) ok = load_a(ma, ma16, mblk * BM, row, left);
          }
      }
      // the copies still in flight land before the CTA exits
      const uint32_t first = af > WG_ASTAGES ? af - WG_ASTAGES : 0;
      for (uint32_t i = first; i < af; ++i)
        mbar_wait_bounded(smem_u32(&afull[i % WG_ASTAGES]),
                          (i / WG_ASTAGES) & 1, nullptr, kDrainNs, p.status,
                          kSiteDrain);
      const uint32_t firstb = bf > WG_BSLOTS ? bf - WG_BSLOTS : 0;
      for (uint32_t i = firstb; i < bf; ++i)
        mbar_wait_bounded(smem_u32(&bfull[i % WG_BSLOTS]),
                          (i / WG_BSLOTS) & 1, nullptr, kDrainNs, p.status,
                          kSiteDrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA
      uint32_t af = 0, bf = 0, qf = 0, tph = 0;
      int slot = 0;
      bool any = false, ok = true;
      auto wait_b = [&](uint32_t i) {
        return mbar_wait_bounded(smem_u32(&bfull[i % WG_BSLOTS]),
                                 (i / WG_BSLOTS) & 1, abort_flag, limit,
                                 p.status, kSiteMmaFull);
      };
      while (ok) {
        const uint32_t qs = qf % WG_QN;
        if (!mbar_wait_bounded(smem_u32(&qfull[qs]), (qf / WG_QN) & 1,
                               abort_flag, limit, p.status, kSiteQueue))
          break;
        const int t = qv[qs];
        mbar_arrive(smem_u32(&qempty[qs]));
        ++qf;
        if (t < 0) break;
        const WTask w = wg_decode(p, t, upre, spoff, NP);
        if (w.rows == 0) continue;
        const int nkb = (w.rows + BK - 1) / BK;
        const int ntile = ((w.nt + 63) / 64) * 64;
        const uint32_t idesc =
            idesc_bf16_f32(BM, ntile) | kAMajorMN | kBMajorMN;
        const uint32_t b0 = bf;  // first B stage of a resident slice
        if (w.res) {
          for (int kb = 0; kb < nkb && ok; ++kb) ok = wait_b(b0 + kb);
          bf += nkb;
        }
        for (int mblk = w.mb0; mblk < w.mb1 && ok; ++mblk) {
          if (!mbar_wait_bounded(smem_u32(&tempty[slot]),
                                 ((tph >> slot) & 1) ^ 1, abort_flag, limit,
                                 p.status, kSiteMmaAcc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + slot * SLOT;
          for (int kb = 0; kb < nkb; ++kb) {
            const uint32_t bi = w.res ? b0 + kb : bf;
            if (!w.res && !wait_b(bi)) {
              ok = false;
              break;
            }
            const uint32_t as = af % WG_ASTAGES;
            if (!mbar_wait_bounded(smem_u32(&afull[as]),
                                   (af / WG_ASTAGES) & 1, abort_flag, limit,
                                   p.status, kSiteMmaFull)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(sA + as * WG_A_BYTES);
            const uint32_t sb = smem_u32(sB + (bi % WG_BSLOTS) * WG_B_BYTES);
            // reduction rows of this stage that belong to the segment (the
            // segment's length is a multiple of 16, or its map ends there)
            const int left = w.rows - kb * BK;
            const int steps = min(BK / UMMA_K, (left + UMMA_K - 1) / UMMA_K);
            for (int kk = 0; kk < steps; ++kk)
              tc_mma_f16(d, sw128_mnmajor_desc(sa + kk * UMMA_K * 128),
                         sw128_mnmajor_desc(sb + kk * UMMA_K * 128), idesc,
                         (kb | kk) != 0);
            any = true;
            tc_commit(smem_u32(&aempty[as]));
            ++af;
            if (!w.res) {
              tc_commit(smem_u32(&bempty[bi % WG_BSLOTS]));
              ++bf;
            }
          }
          if (!ok) break;
          tc_commit(smem_u32(&tfull[slot]));
          tph ^= 1u << slot;
          slot ^= 1;
        }
        if (ok && w.res)
          for (int kb = 0; kb < nkb; ++kb)
            tc_commit(smem_u32(&bempty[(b0 + kb) % WG_BSLOTS]));
      }
      if (any) {
        tc_commit(smem_u32(drain));
        mbar_wait_bounded(smem_u32(drain), 0, nullptr, kDrainNs, p.status,
                          kSiteDrain);
      }
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------- epilogue
    // Each warp owns 32 rows (its TMEM lane quadrant) and half of a block's
    // columns: per 32 columns it writes its rows into a swizzled 4 KB
    // staging tile and one lane issues the TMA store (or reduce-add) of the
    // tile; two tiles alternate, so a tile is rewritten only after its
    // store has read it.
    const int q = warp & 3;
    const int hw = (warp - kEpiWarp0) >> 2;  // which half of the columns
    const int r = q * 32 + lane;
    uint32_t tph = 0, qf = 0;
    int slot = 0;
    int ob = 0;
    bool ok = true;
    uint8_t* stage_base =
        sO + (warp - kEpiWarp0) * WG_OUT_BUFS * WG_OUT_TILE;
    // the gradients stream out once: their lines go first when L2 needs
    // room, so the operand rows (kept with evict_last) stay resident
    const uint64_t pol_out = policy_evict_first();
    while (ok) {
      int t = -1;
      if (lane == 0) {
        const uint32_t qs = qf % WG_QN;
        if (mbar_wait_bounded(smem_u32(&qfull[qs]), (qf / WG_QN) & 1,
                              abort_flag, limit, p.status, kSiteQueue)) {
          t = qv[qs];
          mbar_arrive(smem_u32(&qempty[qs]));
        }
      }
      t = __shfl_sync(0xffffffffu, t, 0);
      ++qf;
      if (t < 0) break;
      const WTask w = wg_decode(p, t, upre, spoff, NP);
      const bool sh = w.seg == 0;
      const int nch = (w.nt + 31) / 32;
      const int c_lo = hw ? (nch + 1) / 2 : 0;
      const int c_hi = hw ? nch : (nch + 1) / 2;
      const CUtensorMap* om = sh ? &p.o_s[w.mat] : &p.o_r[w.mat];
      const int mat_idx = sh ? 0 : w.seg - 1;
      for (int mblk = w.mb0; mblk < w.mb1; ++mblk) {
        const int m0 = mblk * BM;
        if (w.rows == 0) {
          // an expert with no tokens has a zero gradient
          const int row = m0 + r;
          if (!p.accumulate && row < w.M) {
            float* out = p.out_r[w.mat] + (size_t)(w.seg - 1) * w.M * w.N;
            float* orow = out + (size_t)row * w.N + w.n0;
            for (int c = 32 * c_lo; c < min(w.nt, 32 * c_hi); c += 4)
              *reinterpret_cast<float4*>(orow + c) = make_float4(0, 0, 0, 0);
          }
          continue;
        }
        int okw = 0;
        if (lane == 0)
          okw = mbar_wait_bounded(smem_u32(&tfull[slot]), (tph >> slot) & 1,
                                  abort_flag, limit, p.status, kSiteEpilogue);
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ta =
            tmem_base + (static_cast<uint32_t>(q * 32) << 16) + slot * SLOT;
        const int mrow = m0 + q * 32;        // first row of this warp
        // a warp whose rows lie past M (a partial last block) has nothing
        // to store; it skips the staging too, whose buffers the previous
        // block's last stores may still be reading (bulk_wait_read_le1
        // counts only committed stores)
        if (mrow < w.M) {
          for (int c = c_lo; c < c_hi; ++c) {
            uint32_t v[32];
            tmem_ld16(ta + 32 * c,
                      *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
            tmem_ld16(ta + 32 * c + 16,
                      *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
            tmem_ld_wait();
            uint8_t* tile = stage_base + ob * WG_OUT_TILE;
            if (lane == 0) bulk_wait_read_le1();
            __syncwarp();
            // row `lane`: 16-byte chunk k at position k ^ (lane & 7) (the
            // 128-byte swizzle of the tensor map)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t a =
                  smem_u32(tile + lane * 128 + ((k ^ (lane & 7)) * 16));
              asm volatile(
                  "st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                  "r"(v[4 * k]), "r"(v[4 * k + 1]), "r"(v[4 * k + 2]),
                  "r"(v[4 * k + 3])
                  : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (p.accumulate)
                tma_reduce_add_3d(om, smem_u32(tile), w.n0 + 32 * c, mrow,
                                  mat_idx, pol_out);
              else
                tma_store_3d(om, smem_u32(tile), w.n0 + 32 * c, mrow,
                             mat_idx, pol_out);
              bulk_commit();
            }
            ob = (ob + 1) % WG_OUT_BUFS;
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&tempty[slot]));
        tph ^= 1u << slot;
        slot ^= 1;
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

size_t wgrad_smem_bytes(int E) {
  return 1024 + WG_BSLOTS * WG_B_BYTES + WG_ASTAGES * WG_A_BYTES +
         WG_OUT_BYTES + kWgBars * sizeof(uint64_t) + 4 * sizeof(uint32_t) +
         sizeof(int) * (WG_QN + kMats * (E + 1) + 1 + (E + 1));
}

bool token_maps(CUtensorMap (&m)[kTokBoxes], const void* base, uint64_t k,
                uint64_t rows) {
  for (int b = 0; b < kTokBoxes; ++b)
    if (!make_tmap_bf16(&m[b], base, k, rows, 16u << b)) return false;
  return true;
}

}  // namespace

size_t expert_backward_rows_cap(int T, int K, int E) {
  return (size_t)T * K + (size_t)(kPadRows - 1) * E;
}

int launch_expert_backward(const BwdArgs& a, cudaStream_t s) {
  auto mark = [&](int i) {
    if (a.events != nullptr)
      cudaEventRecord(static_cast<cudaEvent_t>(a.events[i]), s);
  };
  const int T = a.T, K = a.topk, E = a.E, H = a.H, I = a.I, Is = a.I_shared;
  const int TK = T * K;
  const int cap = static_cast<int>(expert_backward_rows_cap(T, K, E));
  if (H / 8 > kRowThreads * kMaxVec || E > 1024) return MOE_ERR_UNSUPPORTED;
  if (dgrad_smem_bytes(E) > kSmemLimit || wgrad_smem_bytes(E) > kSmemLimit)
    return MOE_ERR_UNSUPPORTED;
  // ---- padded dispatch
  mark(0);
  bwd_pad_kernel<<<(TK + kPadThreads - 1) / kPadThreads, kPadThreads, 0, s>>>(
      a.topk_idx, a.dest, a.offsets, a.counts, a.gate, TK, E, cap, a.poff,
      a.pdest, a.gp, a.ticket, a.status);
  bwd_gather_kernel<<<T, kRowThreads, 0, s>>>(a.x, a.dout, a.pdest, H, K,
                                              a.xpp, a.dpp);
  bwd_zero_pad_kernel<<<E, kRowThreads, 0, s>>>(a.counts, a.poff, H, a.xpp,
                                                a.dpp, a.gp);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;

  // ---- recompute p, q and g * m
  DgParams rc;
  std::memset(&rc, 0, sizeof(rc));
  bool ok = token_maps(rc.tok_r, a.xpp, H, cap) &&
            token_maps(rc.tok_s, a.x, H, T) &&
            make_tmap_bf16(&rc.wa_r, a.w1, H, (uint64_t)E * I, BM) &&
            make_tmap_bf16(&rc.wb_r, a.w3, H, (uint64_t)E * I, BM) &&
            make_tmap_bf16(&rc.wa_s, a.ws1, H, Is, BM) &&
            make_tmap_bf16(&rc.wb_s, a.ws3, H, Is, BM);
  if (!ok) return MOE_ERR_CUDA;
  rc.poff = a.poff;
  rc.gp = a.gp;
  rc.p_r = a.p_r;
  rc.q_r = a.q_r;
  rc.p_s = a.p_s;
  rc.q_s = a.q_s;
  rc.hg_r = a.hg_r;
  rc.hg_s = a.hg_s;
  rc.status = a.status;
  rc.wait_limit_ns = a.wait_limit_ns;
  rc.E = E;
  rc.T = T;
  rc.TKP = cap;
  rc.n_r = I;
  rc.n_s = Is;
  rc.k_r = H;
  rc.k_s = H;
  rc.wrows_r = I;
  mark(1);
  int rcode = launch_dgrad<kRecomp>(rc, s);
  if (rcode != MOE_OK) return rcode;

  // ---- D = dout W2 (per segment), dgate partials, dp, dq
  DgParams dd;
  std::memset(&dd, 0, sizeof(dd));
  ok = token_maps(dd.tok_r, a.dpp, H, cap) &&
       token_maps(dd.tok_s, a.dout, H, T) &&
       make_tmap_bf16(&dd.wa_r, a.w2, I, (uint64_t)E * H, BK) &&
       make_tmap_bf16(&dd.wa_s, a.ws2, Is, H, BK);
  if (!ok) return MOE_ERR_CUDA;
  dd.wb_r = dd.wa_r;
  dd.wb_s = dd.wa_s;
  dd.poff = a.poff;
  dd.gp = a.gp;
  dd.p_r = a.p_r;
  dd.q_r = a.q_r;
  dd.p_s = a.p_s;
  dd.q_s = a.q_s;
  dd.dp_r = a.dp_r;
  dd.dq_r = a.dq_r;
  dd.dp_s = a.dp_s;
  dd.dq_s = a.dq_s;
  dd.dgp = a.dgp;
  dd.status = a.status;
  dd.wait_limit_ns = a.wait_limit_ns;
  dd.E = E;
  dd.T = T;
  dd.TKP = cap;
  dd.n_r = I;
  dd.n_s = Is;
  dd.k_r = H;
  dd.k_s = H;
  dd.wrows_r = H;
  dd.nfb = (I + 2 * BM - 1) / (2 * BM);
  mark(2);
  rcode = launch_dgrad<kDgradDown>(dd, s);
  if (rcode != MOE_OK) return rcode;

  // ---- dxpp = dp W1 + dq W3 (per segment), dxs likewise
  DgParams du;
  std::memset(&du, 0, sizeof(du));
  ok = token_maps(du.tok_r, a.dp_r, I, cap) &&
       token_maps(du.tok_s, a.dp_s, Is, T) &&
       token_maps(du.tok2_r, a.dq_r, I, cap) &&
       token_maps(du.tok2_s, a.dq_s, Is, T) &&
       make_tmap_bf16(&du.wa_r, a.w1, H, (uint64_t)E * I, BK) &&
       make_tmap_bf16(&du.wb_r, a.w3, H, (uint64_t)E * I, BK) &&
       make_tmap_bf16(&du.wa_s, a.ws1, H, Is, BK) &&
       make_tmap_bf16(&du.wb_s, a.ws3, H, Is, BK);
  if (!ok) return MOE_ERR_CUDA;
  du.poff = a.poff;
  du.gp = a.gp;
  du.out_r = a.dxpp;
  du.out_s = a.dxs;
  du.status = a.status;
  du.wait_limit_ns = a.wait_limit_ns;
  du.E = E;
  du.T = T;
  du.TKP = cap;
  du.n_r = H;
  du.n_s = H;
  du.k_r = 2 * I;
  du.k_s = 2 * Is;
  du.wrows_r = I;
  mark(3);
  rcode = launch_dgrad<kDgradUp>(du, s);
  if (rcode != MOE_OK) return rcode;

  // ---- weight gradients
  WgParams wp;
  std::memset(&wp, 0, sizeof(wp));
  ok = make_tmap_bf16(&wp.a_r[0], a.dp_r, I, cap, BK) &&
       make_tmap_bf16(&wp.a_r[1], a.dq_r, I, cap, BK) &&
       make_tmap_bf16(&wp.a_r[2], a.dpp, H, cap, BK) &&
       make_tmap_bf16(&wp.b_r[0], a.xpp, H, cap, BK) &&
       make_tmap_bf16(&wp.b_r[1], a.xpp, H, cap, BK) &&
       make_tmap_bf16(&wp.b_r[2], a.hg_r, I, cap, BK) &&
       make_tmap_bf16(&wp.a_s[0], a.dp_s, Is, T, BK) &&
       make_tmap_bf16(&wp.a_s[1], a.dq_s, Is, T, BK) &&
       make_tmap_bf16(&wp.a_s[2], a.dout, H, T, BK) &&
       make_tmap_bf16(&wp.b_s[0], a.x, H, T, BK) &&
       make_tmap_bf16(&wp.b_s[1], a.x, H, T, BK) &&
       make_tmap_bf16(&wp.b_s[2], a.hg_s, Is, T, BK) &&
       make_tmap_bf16(&wp.a_r16[0], a.dp_r, I, cap, 16) &&
       make_tmap_bf16(&wp.a_r16[1], a.dq_r, I, cap, 16) &&
       make_tmap_bf16(&wp.a_r16[2], a.dpp, H, cap, 16) &&
       make_tmap_bf16(&wp.b_r16[0], a.xpp, H, cap, 16) &&
       make_tmap_bf16(&wp.b_r16[1], a.xpp, H, cap, 16) &&
       make_tmap_bf16(&wp.b_r16[2], a.hg_r, I, cap, 16) &&
       make_tmap_bf16(&wp.a_s16[0], a.dp_s, Is, T, 16) &&
       make_tmap_bf16(&wp.a_s16[1], a.dq_s, Is, T, 16) &&
       make_tmap_bf16(&wp.a_s16[2], a.dout, H, T, 16) &&
       make_tmap_bf16(&wp.b_s16[0], a.x, H, T, 16) &&
       make_tmap_bf16(&wp.b_s16[1], a.x, H, T, 16) &&
       make_tmap_bf16(&wp.b_s16[2], a.hg_s, Is, T, 16);
  ok = ok && make_tmap_f32_3d_store(&wp.o_r[0], a.dw1, H, I, E) &&
       make_tmap_f32_3d_store(&wp.o_r[1], a.dw3, H, I, E) &&
       make_tmap_f32_3d_store(&wp.o_r[2], a.dw2, I, H, E) &&
       make_tmap_f32_3d_store(&wp.o_s[0], a.dws1, H, Is, 1) &&
       make_tmap_f32_3d_store(&wp.o_s[1], a.dws3, H, Is, 1) &&
       make_tmap_f32_3d_store(&wp.o_s[2], a.dws2, Is, H, 1);
  if (!ok) return MOE_ERR_CUDA;
  wp.poff = a.poff;
  wp.ticket = a.ticket;
  wp.out_r[0] = a.dw1;
  wp.out_r[1] = a.dw3;
  wp.out_r[2] = a.dw2;
  wp.out_s[0] = a.dws1;
  wp.out_s[1] = a.dws3;
  wp.out_s[2] = a.dws2;
  wp.status = a.status;
  wp.wait_limit_ns = a.wait_limit_ns;
  wp.E = E;
  wp.T = T;
  wp.TKP = cap;
  wp.H = H;
  wp.I = I;
  wp.Is = Is;
  wp.accumulate = a.accumulate;
  {
    const size_t smem = wgrad_smem_bytes(E);
    if (cudaFuncSetAttribute(wgrad_gemm_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MOE_ERR_CUDA;
    mark(4);
    wgrad_gemm_kernel<<<gemm_ctas(), kWgThreads, smem, s>>>(wp);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }

  // ---- token gradient and gate gradients
  mark(5);
  bwd_finalize_kernel<<<T, kRowThreads, 0, s>>>(
      a.dout, a.dxs, a.dxpp, a.pdest, a.dgp, dd.nfb, H, K, a.dx, a.dgate);
  mark(6);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
