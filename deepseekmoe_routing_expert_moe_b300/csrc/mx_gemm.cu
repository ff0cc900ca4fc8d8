// FP8 (E4M3) grouped expert GEMMs with power-of-two group scales applied by
// the sm_103a tensor cores.
//
// "02 · DeepSeek-V3" (PaperTrace) §2 quantizes activations per 1 x 128 tile
// and weights per 128 x 128 block and promotes every 128-element slice of
// the reduction, scaled, into fp32 on the CUDA cores; it likens the groups
// to the microscaling formats whose scaling Blackwell's tensor cores apply
// themselves.  That is this file: with every scale a power of two (a UE8M0
// byte, 2^(b - 127)), tcgen05.mma kind::mxf8f6f4.block_scale multiplies each
// 32-element slice of a product by its row's and its column's scale inside
// the tensor core and accumulates in fp32 tensor memory, so no partial sum
// leaves the tensor memory before the unit's end and nothing is promoted on
// the CUDA cores.  A 128-element group is four such slices with the same
// scale.
//
//   up   (kMxUp):   m = silu(A W1^T) * (A W3^T), quantized again to E4M3
//                   per 1 x 128 tile with power-of-two scales
//   down (kMxDown): y = M W2^T, stored as bf16
//
// Orientation and work list as the BF16 kernels (grouped_gemm.cu): weights
// are the MMA's M side (128 rows = one scale block), tokens its N side; a
// unit is (segment, feature block, chunk of rows); one persistent CTA per
// SM, 11 warps:
//   warp 0 lane 0   weight producer: per 128-wide k-block the two 128 x 128
//                   E4M3 tiles, 128-byte swizzle, a deep ring (HBM stream)
//   warp 2          token producer: per k-block the scale atoms (below) and
//                   the chunk's token tile (boxes of 128/64/32/16 rows)
//   warp 1 lane 0   MMA: tcgen05.cp of the k-block's scale atoms into
//                   tensor memory, then 4 block-scaled MMAs (K = 32) per
//                   accumulator, slice j reading byte j of each scale word
//   warps 3..10     epilogue, two warps per tensor-memory lane quadrant,
//                   each with half of the unit's 16-column chunks:
//                   tcgen05.ld, then (up) SwiGLU into fp32 registers and
//                   each column's max over the warp's 32 feature rows; the
//                   tensor memory is released at once, and after one
//                   barrier every column's 1 x 128 tile maximum (the four
//                   quadrants' maxima) gives its power-of-two scale and the
//                   codes; (down) bf16 conversion and stores
// Scale atoms (the layout tcgen05.cp 32x128b.warpx4 copies into the four
// lane quadrants): 512 bytes for 128 rows (or columns) r, 4 bytes j per row
// at byte (r % 32) * 16 + (r / 32) * 4 + j; an MMA slice reads byte j = its
// scale ID.  A group scale is the same for the four 32-element slices of
// its k-block, so byte j holds the scale of k-block 4g + j and the four
// k-blocks of group g share one atom set (every slice of k-block kb reads
// byte kb % 4): one atom per weight tile and one per 128 token columns,
// built and copied once per four k-blocks.
// Tensor memory: two accumulator slots of 232 columns (a unit with N <= 112
// puts both accumulators in one slot, so consecutive units alternate slots
// and the epilogue of one overlaps the MMAs of the next; a wider unit takes
// both), and two sets of 24 scale columns from column 464.
// Every wait is bounded (MOE_ERR_TIMEOUT in the status word, then a clean
// exit: in-flight copies and MMAs are drained, tensor memory is freed).
#include <cuda.h>
#include <cuda_fp8.h>

#include <cstdint>
#include <cstring>

#include "device_common.cuh"
#include "internal.h"
#include "unit_list.cuh"

namespace moe {
namespace {

constexpr int XM = 128;       // weight rows per tile = MMA M = scale block
constexpr int XK = 128;       // k per stage: 128 E4M3 = one 128 B row
constexpr int XUMMA_K = 32;   // k of one block-scaled MMA (one scale)
constexpr uint32_t XW_BYTES = XM * XK;      // one weight tile, 16 KB
constexpr uint32_t XWSTAGE = 2 * XW_BYTES;  // both weight tiles
constexpr uint32_t XSF_BYTES = 2048;        // atoms: W tile a, b, tokens x2
constexpr int XSF_RING = 4;    // atom groups in shared memory
constexpr int XGROUP = 4;      // k-blocks per atom group (one byte each)
constexpr int XSLOT = 232;                  // accumulator slot columns
constexpr int XNARROW = 112;  // widest N with both accumulators in a slot
constexpr int XSF_COL0 = 464;               // scale sets: 464, 488
constexpr int XSF_SET = 24;
constexpr uint32_t XTMEM_COLS = 512;
constexpr int XTOK_BOXES = 4;               // token boxes of 16..128 rows
constexpr int XEPI0 = 3;                    // first epilogue warp
constexpr int XEPI = 8;  // two per lane quadrant, half the columns each
constexpr int XTHREADS = 32 * (XEPI0 + XEPI);
constexpr size_t XSMEM_LIMIT = 232448;      // 227 KB per CTA
constexpr uint64_t XDRAIN_NS = 2000000000ull;

enum { kMxUp = 0, kMxDown = 1 };
enum {
  kMxSiteProducer = 51,
  kMxSiteMmaAcc = 52,
  kMxSiteMmaFull = 53,
  kMxSiteEpilogue = 54,
  kMxSiteDrain = 55,
  kMxSiteOffsets = 56
};

// NT largest token chunk (MMA N), WS weight ring depth, TS token ring depth
template <int NT_, int WS_, int TS_>
struct MxPipe {
  static constexpr int NT = NT_;
  static constexpr int WS = WS_;
  static constexpr int TS = TS_;
};
using MxStream = MxPipe<192, 4, 3>;   // mean rows per expert < 256
using MxCompute = MxPipe<224, 4, 2>;  // mean rows per expert >= 256
constexpr int kMxComputeRows = 256;

template <class P>
struct MxRing {
  static constexpr uint32_t TSTAGE = P::NT * XK;  // token tile bytes
  static constexpr uint32_t BYTES =
      P::WS * XWSTAGE + P::TS * TSTAGE + XSF_RING * XSF_BYTES;
  static constexpr int BARS = 2 * P::WS + 2 * P::TS + 5;
  static constexpr uint32_t RED = 2 * 4 * P::NT * sizeof(float);
  static_assert(P::NT % 16 == 0 && P::NT <= 2 * XNARROW, "chunk");
  static_assert(TSTAGE % 1024 == 0, "swizzle atoms stay aligned");
};

struct MxParams {  // CUtensorMap members carry their 64-byte alignment
  CUtensorMap tok_routed[XTOK_BOXES];  // up: xpq [TK, H]   down: mq [TK, I]
  CUtensorMap tok_shared[XTOK_BOXES];  // up: xq [T, H]     down: msq [T, I_s]
  CUtensorMap wa_routed;  // up: w1 [E*I, H]    down: w2 [E*H, I]
  CUtensorMap wb_routed;  // up: w3 [E*I, H]    down: w2 (rows + 128)
  CUtensorMap wa_shared;  // up: ws1 [I_s, H]   down: ws2 [H, I_s]
  CUtensorMap wb_shared;  // up: ws3 [I_s, H]   down: ws2 (rows + 128)
  const uint8_t* ts_routed;  // token scales [TK, K/128]
  const uint8_t* ts_shared;  // [T, K/128]
  const uint8_t* sa_routed;  // block scales of tile a [rows/128, K/128]
  const uint8_t* sb_routed;  // of tile b (up: W3; down: W2)
  const uint8_t* sa_shared;
  const uint8_t* sb_shared;
  const int32_t* offsets;    // [E+1]
  uint8_t* q_routed;         // up: m codes [TK, I]
  uint8_t* qs_routed;        // up: m scales [TK, I/128]
  uint8_t* q_shared;         // up: [T, I_s]
  uint8_t* qs_shared;        // up: [T, I_s/128]
  uint16_t* y_routed;        // down: yp [TK, H]
  uint16_t* y_shared;        // down: ys [T, H]
  DevStatus* status;
  unsigned long long wait_limit_ns;
  int E, T, TK;
  int n_routed, n_shared;  // output features of a routed / the shared one
  int k_routed, k_shared;  // reduction length of a routed / the shared one
};

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A and B
// E4M3 (format 0), K-major, dense, D f32, scales UE8M0 (bit 23), shape
// M x N (N/8 at bit 17, M/16 at bit 24); the scale slice IDs (which byte of
// each 32-bit scale word a slice reads) at bits 29-30 (A) and 4-5 (B).
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int M, int N) {
  return (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_slice(uint32_t base, int k) {
  return base | (static_cast<uint32_t>(k) << 4) |
         (static_cast<uint32_t>(k) << 29);
}

// D[tmem] (+)= (A * sA) (B * sB)^T over one K = 32 slice
__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t a_desc,
                                          uint64_t b_desc, uint32_t idesc,
                                          uint32_t sfa_tmem,
                                          uint32_t sfb_tmem,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
      "r"(accumulate)
      : "memory");
}

// Shared-memory descriptor of one scale atom: 32 rows of 16 bytes, 8-row
// groups 128 bytes apart, no swizzle.
__device__ __forceinline__ uint64_t atom_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128u >> 4) << 16;  // LBO
  d |= static_cast<uint64_t>(128u >> 4) << 32;  // SBO
  d |= static_cast<uint64_t>(1u) << 46;         // descriptor version
  return d;
}

// one atom into the four lane quadrants of tensor memory at `taddr`
__device__ __forceinline__ void tc_cp_atom(uint32_t taddr, uint32_t smem) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(
                   taddr),
               "l"(atom_desc(smem))
               : "memory");
}

__device__ __forceinline__ uint32_t e4m3_of(float v) {
  return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// named barrier of the four epilogue warps
__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * XEPI) : "memory");
}

template <int MODE, class P>
__global__ void __launch_bounds__(XTHREADS, 1)
    mx_gemm_kernel(const __grid_constant__ MxParams p) {
  constexpr int FB = (MODE == kMxUp) ? XM : 2 * XM;
  constexpr int NT = P::NT, kWStages = P::WS, kTStages = P::TS;
  constexpr uint32_t TSTAGE = MxRing<P>::TSTAGE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;                              // weight ring
  uint8_t* sT = smem + kWStages * XWSTAGE;         // token ring
  uint8_t* sF = sT + kTStages * TSTAGE;            // scale atoms per stage
  float* s_red = reinterpret_cast<float*>(sF + XSF_RING * XSF_BYTES);
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + MxRing<P>::BYTES + MxRing<P>::RED);
  uint64_t* wfull = bars;
  uint64_t* wempty = wfull + kWStages;
  uint64_t* kfull = wempty + kWStages;
  uint64_t* kempty = kfull + kTStages;
  uint64_t* tfull = kempty + kTStages;  // per TMEM slot
  uint64_t* tempty = tfull + 2;         // per TMEM slot
  uint64_t* drain = tempty + 2;
  volatile uint32_t* misc =
      reinterpret_cast<volatile uint32_t*>(bars + MxRing<P>::BARS);
  // misc[0] TMEM base, [1] abort flag, [2] bad offsets, [3..4] the
  // epilogue warps' failure words of even / odd units
  const int E = p.E;
  const int NS = E + 1;
  int* useg = reinterpret_cast<int*>(const_cast<uint32_t*>(misc) + 8);
  int* srows = useg + NS + 1;
  int* srow0 = srows + NS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kWStages; ++i) {
      mbar_init(smem_u32(&wfull[i]), 1);
      mbar_init(smem_u32(&wempty[i]), 1);
    }
    for (int i = 0; i < kTStages; ++i) {
      mbar_init(smem_u32(&kfull[i]), 1);
      mbar_init(smem_u32(&kempty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), 32 * XEPI);
    }
    mbar_init(smem_u32(drain), 1);
    misc[1] = 0;
    misc[2] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
#pragma unroll
    for (int b = 0; b < XTOK_BOXES; ++b) {
      prefetch_tmap(&p.tok_routed[b]);
      prefetch_tmap(&p.tok_shared[b]);
    }
    prefetch_tmap(&p.wa_routed);
    prefetch_tmap(&p.wb_routed);
    prefetch_tmap(&p.wa_shared);
    prefetch_tmap(&p.wb_shared);
  }
  if (warp == 2) {
    // segment table: rows, first row, and the exclusive prefix of units
    const int nfb_r = (p.n_routed + FB - 1) / FB;
    const int nfb_s = (p.n_shared + FB - 1) / FB;
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
    tmem_alloc(smem_u32(const_cast<uint32_t*>(&misc[0])), XTMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  int total = useg[NS];
  if (misc[2]) {
    if (threadIdx.x == 0)
      record_error(p.status, MOE_ERR_DEVICE_BOUNDS, kMxSiteOffsets);
    total = 0;
  }
  const uint64_t limit = p.wait_limit_ns;

  if (warp == 0) {
    if (lane == 0) {
      // ----------------------------------------------- weight producer
      uint32_t stage = 0, phase = 0, issued = 0;
      const uint64_t pol_w = policy_evict_first();
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const Unit w = decode_unit<NT>(u, useg, srow0, srows, NS);
        const bool sh = (w.seg == 0);
        const CUtensorMap* wa = sh ? &p.wa_shared : &p.wa_routed;
        const CUtensorMap* wb = sh ? &p.wb_shared : &p.wb_routed;
        const int wrow = (sh ? 0 : (w.seg - 1) * p.n_routed) + w.f * FB;
        const int wrow_b = (MODE == kMxUp) ? wrow : wrow + XM;
        const int nkb = (sh ? p.k_shared : p.k_routed) / XK;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&wempty[stage]), phase ^ 1,
                                 abort_flag, limit, p.status,
                                 kMxSiteProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&wfull[stage]);
          uint8_t* st = sW + stage * XWSTAGE;
          mbar_arrive_expect_tx(fb, XWSTAGE);
          tma_load_2d_hint(smem_u32(st), wa, kb * XK, wrow, fb, pol_w);
          tma_load_2d_hint(smem_u32(st + XW_BYTES), wb, kb * XK, wrow_b, fb,
                           pol_w);
          ++issued;
          if (++stage == kWStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      // drain: the last min(issued, stages) loads must land before exit
      const uint32_t first = issued > kWStages ? issued - kWStages : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait_bounded(smem_u32(&wfull[i % kWStages]),
                          (i / kWStages) & 1, nullptr, XDRAIN_NS, p.status,
                          kMxSiteDrain);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------ scale atoms + token producer
    uint32_t stage = 0, phase = 0, issued = 0, sfg = 0;
    const uint64_t pol_t = policy_evict_last();
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const Unit w = decode_unit<NT>(u, useg, srow0, srows, NS);
      const bool sh = (w.seg == 0);
      const CUtensorMap* tok = sh ? p.tok_shared : p.tok_routed;
      const int nkb = (sh ? p.k_shared : p.k_routed) / XK;
      const int nout = sh ? p.n_shared : p.n_routed;
      const uint8_t* ts = sh ? p.ts_shared : p.ts_routed;
      const uint8_t* sa = sh ? p.sa_shared : p.sa_routed;
      const uint8_t* sb = sh ? p.sb_shared : p.sb_routed;
      const int wrow = (sh ? 0 : (w.seg - 1) * nout) + w.f * FB;
      const int blk_a = wrow / XM;
      const int blk_b = (MODE == kMxUp) ? blk_a : blk_a + 1;
      // the down projection's second tile may lie past the expert's rows
      // (its outputs are not stored): scale 1 there
      const bool b_live = (MODE == kMxUp) || (w.f * FB + XM < nout);
      const uint32_t tx = (uint32_t)w.n * XK;
      // the scale words of k-block group g (byte j: k-block 4g + j): weight
      // tiles a, b and token rows lane + 32 c (c < 8: columns 0..255); 127
      // (scale 1) past the chunk or past the last k-block; fetched one
      // group ahead of their atoms
      const bool word_loads = (nkb % XGROUP) == 0;
      auto word = [&](const uint8_t* base, size_t at, int kb0) -> uint32_t {
        if (word_loads)
          return __ldg(reinterpret_cast<const uint32_t*>(base + at + kb0));
        uint32_t v = 0;
#pragma unroll
        for (int j = 0; j < XGROUP; ++j)
          v |= (kb0 + j < nkb ? (uint32_t)__ldg(base + at + kb0 + j) : 127u)
               << (8 * j);
        return v;
      };
      auto fetch = [&](int g, uint32_t (&v)[10]) {
        const int kb0 = g * XGROUP;
        if (kb0 >= nkb) {
#pragma unroll
          for (int i = 0; i < 10; ++i) v[i] = 0x7F7F7F7Fu;
          return;
        }
        v[0] = word(sa, (size_t)blk_a * nkb, kb0);
        v[1] = b_live ? word(sb, (size_t)blk_b * nkb, kb0) : 0x7F7F7F7Fu;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int n = 32 * c + lane;
          v[2 + c] = n < w.rows ? word(ts, (size_t)(w.row0 + n) * nkb, kb0)
                                : 0x7F7F7F7Fu;
        }
      };
      uint32_t v0[10], v1[10];
      fetch(0, v0);
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        int okw = 1;
        if (lane == 0)
          okw = mbar_wait_bounded(smem_u32(&kempty[stage]), phase ^ 1,
                                  abort_flag, limit, p.status,
                                  kMxSiteProducer);
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) {
          ok = false;
          break;
        }
        if (kb % XGROUP == 0) {
          // a new group: its atoms into ring entry sfg % XSF_RING (the
          // entry's previous group started >= XSF_RING k-blocks ago, so
          // the kempty wait above has seen its copies complete)
          fetch(kb / XGROUP + 1, v1);
          uint8_t* sf = sF + (sfg % XSF_RING) * XSF_BYTES;
          reinterpret_cast<uint4*>(sf)[lane] =
              make_uint4(v0[0], v0[0], v0[0], v0[0]);
          reinterpret_cast<uint4*>(sf + 512)[lane] =
              make_uint4(v0[1], v0[1], v0[1], v0[1]);
          // token columns 128 t .. 128 t + 127: lane holds rows lane + 32 c
          reinterpret_cast<uint4*>(sf + 1024)[lane] =
              make_uint4(v0[2], v0[3], v0[4], v0[5]);
          if (w.n > 128)
            reinterpret_cast<uint4*>(sf + 1536)[lane] =
                make_uint4(v0[6], v0[7], v0[8], v0[9]);
#pragma unroll
          for (int i = 0; i < 10; ++i) v0[i] = v1[i];
          ++sfg;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const uint32_t fb = smem_u32(&kfull[stage]);
          uint8_t* stok = sT + stage * TSTAGE;
          mbar_arrive_expect_tx(fb, tx);
          // token rows [row0, row0 + n) as boxes of 128/64/32/16 rows
          int off = 0;
#pragma unroll
          for (int b = XTOK_BOXES - 1; b >= 0; --b) {
            if ((w.n >> 4) & (1 << b)) {
              tma_load_2d_hint(smem_u32(stok + off * XK), &tok[b], kb * XK,
                               w.row0 + off, fb, pol_t);
              off += 16 << b;
            }
          }
        }
        ++issued;
        if (++stage == kTStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
    }
    if (lane == 0) {
      const uint32_t first = issued > kTStages ? issued - kTStages : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait_bounded(smem_u32(&kfull[i % kTStages]),
                          (i / kTStages) & 1, nullptr, XDRAIN_NS, p.status,
                          kMxSiteDrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA
      uint32_t wstage = 0, wphase = 0, kstage = 0, kphase = 0;
      uint32_t tph = 0;  // bit s: parity of the uses of TMEM slot s so far
      uint32_t sfg = 0;  // atom groups copied so far
      int slot = 0;
      bool any = false;
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const Unit w = decode_unit<NT>(u, useg, srow0, srows, NS);
        const int nkb = ((w.seg == 0) ? p.k_shared : p.k_routed) / XK;
        const bool wide = w.n > XNARROW;
        const int s1 = wide ? (slot ^ 1) : slot;
        if (!mbar_wait_bounded(smem_u32(&tempty[slot]),
                               ((tph >> slot) & 1) ^ 1, abort_flag, limit,
                               p.status, kMxSiteMmaAcc))
          break;
        if (wide && !mbar_wait_bounded(smem_u32(&tempty[s1]),
                                       ((tph >> s1) & 1) ^ 1, abort_flag,
                                       limit, p.status, kMxSiteMmaAcc))
          break;
        tc_fence_after();
        const uint32_t da = tmem_base + slot * XSLOT;
        const uint32_t db = wide ? tmem_base + s1 * XSLOT : da + XNARROW;
        const uint32_t idesc = idesc_mx_e4m3(XM, w.n);
        bool ok = true;
        uint32_t sfc = 0;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&wfull[wstage]), wphase,
                                 abort_flag, limit, p.status,
                                 kMxSiteMmaFull) ||
              !mbar_wait_bounded(smem_u32(&kfull[kstage]), kphase,
                                 abort_flag, limit, p.status,
                                 kMxSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (kb % XGROUP == 0) {
            // the group's atoms (written before this k-block's kfull
            // arrive) into one of two tensor-memory scale sets
            sfc = tmem_base + XSF_COL0 + XSF_SET * (sfg & 1);
            const uint32_t sf = smem_u32(sF + (sfg % XSF_RING) * XSF_BYTES);
            tc_cp_atom(sfc, sf);               // weight tile a
            tc_cp_atom(sfc + 8, sf + 512);     // weight tile b
            tc_cp_atom(sfc + 16, sf + 1024);   // token columns 0..127
            if (w.n > 128) tc_cp_atom(sfc + 20, sf + 1536);  // 128..
            ++sfg;
          }
          const uint32_t s0 = smem_u32(sW + wstage * XWSTAGE);
          const uint32_t st = smem_u32(sT + kstage * TSTAGE);
          // every slice of this k-block reads byte kb % 4 of the atoms
          const uint32_t id = idesc_slice(idesc, kb % XGROUP);
#pragma unroll
          for (int kk = 0; kk < XK / XUMMA_K; ++kk) {
            const uint64_t bdesc = sw128_kmajor_desc(st + kk * XUMMA_K);
            const uint32_t acc = (kb | kk) != 0;
            tc_mma_mx(da, sw128_kmajor_desc(s0 + kk * XUMMA_K), bdesc, id,
                      sfc, sfc + 16, acc);
            tc_mma_mx(db, sw128_kmajor_desc(s0 + XW_BYTES + kk * XUMMA_K),
                      bdesc, id, sfc + 8, sfc + 16, acc);
          }
          any = true;
          tc_commit(smem_u32(&wempty[wstage]));
          tc_commit(smem_u32(&kempty[kstage]));
          if (++wstage == kWStages) {
            wstage = 0;
            wphase ^= 1;
          }
          if (++kstage == kTStages) {
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
      if (any) {  // every issued MMA completes before TMEM is released
        tc_commit(smem_u32(drain));
        mbar_wait_bounded(smem_u32(drain), 0, nullptr, XDRAIN_NS, p.status,
                          kMxSiteDrain);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- epilogue
    constexpr int MC = (NT / 16 + 1) / 2;  // chunks of one half, at most
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int half = (warp - XEPI0) >> 2;
    const int r = q * 32 + lane;
    const int et = threadIdx.x - 32 * XEPI0;
    uint32_t tph = 0;
    int slot = 0, it = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++it) {
      const Unit w = decode_unit<NT>(u, useg, srow0, srows, NS);
      const bool wide = w.n > XNARROW;
      const int s1 = wide ? (slot ^ 1) : slot;
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait_bounded(smem_u32(&tfull[slot]), (tph >> slot) & 1,
                               abort_flag, limit, p.status, kMxSiteEpilogue);
        if (ok && wide)
          ok = mbar_wait_bounded(smem_u32(&tfull[s1]), (tph >> s1) & 1,
                                 abort_flag, limit, p.status,
                                 kMxSiteEpilogue);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // the unit's vote: every epilogue warp stops together (they meet at
      // named barriers below), none is left waiting at one
      {
        volatile uint32_t* fw = misc + 3 + (it & 1);
        if (et == 0) *fw = 0;
        epi_bar();
        if (!ok && lane == 0) *fw = 1;
        epi_bar();
        if (*fw) break;
      }
      tc_fence_after();
      const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
      const uint32_t ta = tmem_base + lane_off + slot * XSLOT;
      const uint32_t tb =
          wide ? tmem_base + lane_off + s1 * XSLOT : ta + XNARROW;
      const bool sh = (w.seg == 0);
      const int nout = sh ? p.n_shared : p.n_routed;
      // this warp's chunks [c_lo, c_hi) of the unit's n / 16
      const int nch = w.n >> 4;
      const int c_lo = half ? (nch + 1) >> 1 : 0;
      const int c_hi = half ? nch : (nch + 1) >> 1;
      auto release = [&](int sl) {
        tc_fence_before();
        mbar_arrive(smem_u32(&tempty[sl]));
      };
      if (MODE == kMxUp) {
        float* red = s_red + (it & 1) * 4 * NT;
        float m[MC][16];
#pragma unroll
        for (int i = 0; i < MC; ++i) {
          const int c = c_lo + i;
          if (c < c_hi) {
            uint32_t a[16], b[16];
            tmem_ld16(ta + 16 * c, a);
            tmem_ld16(tb + 16 * c, b);
            tmem_ld_wait();
            uint32_t mine = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              m[i][j] = silu_f(__uint_as_float(a[j])) * __uint_as_float(b[j]);
              // |m| bit patterns order like the values
              const uint32_t mx = __reduce_max_sync(
                  0xffffffffu, __float_as_uint(fabsf(m[i][j])));
              if (lane == j) mine = mx;
            }
            if (lane < 16)
              red[q * NT + 16 * c + lane] = __uint_as_float(mine);
          }
        }
        release(slot);
        if (wide) release(s1);
        epi_bar();
        uint8_t* qo = (sh ? p.q_shared : p.q_routed) +
                      (size_t)w.row0 * nout + w.f * XM + r;
        uint8_t* qs = (sh ? p.qs_shared : p.qs_routed) +
                      (size_t)w.row0 * (nout / XM) + w.f;
#pragma unroll
        for (int i = 0; i < MC; ++i) {
          const int c = c_lo + i;
          if (c < c_hi) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = 16 * c + j;
              const float amax =
                  fmaxf(fmaxf(red[col], red[NT + col]),
                        fmaxf(red[2 * NT + col], red[3 * NT + col]));
              const int e = ue8m0_exponent(amax);
              if (col < w.rows) {
                qo[(size_t)col * nout] =
                    (uint8_t)e4m3_of(m[i][j] * pow2_neg(e));
                if (r == j) qs[(size_t)col * (nout / XM)] = (uint8_t)(e + 127);
              }
            }
          }
        }
      } else {
        // every column of this warp's chunks into bf16 pairs first, so the
        // tensor memory goes back to the MMA before the scattered stores
        uint32_t pa[MC][8], pb[MC][8];
#pragma unroll
        for (int i = 0; i < MC; ++i) {
          const int c = c_lo + i;
          if (c < c_hi) {
            uint32_t a[16], b[16];
            tmem_ld16(ta + 16 * c, a);
            tmem_ld16(tb + 16 * c, b);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              pa[i][j] = pack_bf16x2(__uint_as_float(a[2 * j]),
                                     __uint_as_float(a[2 * j + 1]));
              pb[i][j] = pack_bf16x2(__uint_as_float(b[2 * j]),
                                     __uint_as_float(b[2 * j + 1]));
            }
          }
        }
        release(slot);
        if (wide) release(s1);
        uint16_t* out = (sh ? p.y_shared : p.y_routed) +
                        (size_t)w.row0 * nout + w.f * FB + r;
        const bool live_b = w.f * FB + XM + r < nout;
#pragma unroll
        for (int i = 0; i < MC; ++i) {
          const int c = c_lo + i;
          if (c < c_hi) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int row = 16 * c + j;
              if (row < w.rows) {
                uint16_t* o = out + (size_t)row * nout;
                const int sh16 = (j & 1) * 16;
                o[0] = (uint16_t)(pa[i][j >> 1] >> sh16);
                if (live_b) o[XM] = (uint16_t)(pb[i][j >> 1] >> sh16);
              }
            }
          }
        }
      }
      tph ^= 1u << slot;
      if (wide)
        tph ^= 1u << s1;
      else
        slot ^= 1;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, XTMEM_COLS);
  }
}

template <class P>
size_t mx_smem_bytes(int E) {
  return 1024 + MxRing<P>::BYTES + MxRing<P>::RED +
         MxRing<P>::BARS * sizeof(uint64_t) + 8 * sizeof(uint32_t) +
         sizeof(int) * (3 * (E + 1) + 1);
}

template <int MODE, class P>
int mx_launch_shape(const MxParams& mp, cudaStream_t s) {
  auto kern = mx_gemm_kernel<MODE, P>;
  const size_t smem = mx_smem_bytes<P>(mp.E);
  if (smem > XSMEM_LIMIT) return MOE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  kern<<<gemm_ctas(), XTHREADS, smem, s>>>(mp);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// the pipeline shape for this launch's mean rows per routed expert; the
// streaming shape's deeper rings do not fit beside the segment tables of
// the largest expert counts (E = 1024), and the compute shape, correct at
// any rows per expert, serves those
template <int MODE>
int mx_launch(const MxParams& mp, cudaStream_t s) {
  const long long mean_rows = mp.E > 0 ? (long long)mp.TK / mp.E : 0;
  const bool stream = mean_rows < kMxComputeRows &&
                      mx_smem_bytes<MxStream>(mp.E) <= XSMEM_LIMIT;
  return stream ? mx_launch_shape<MODE, MxStream>(mp, s)
                : mx_launch_shape<MODE, MxCompute>(mp, s);
}

// token-operand maps of one [rows, k] E4M3 tensor, boxes of 16..128 rows
bool mx_token_maps(CUtensorMap (&m)[XTOK_BOXES], const void* base,
                   uint64_t k, uint64_t rows) {
  for (int b = 0; b < XTOK_BOXES; ++b)
    if (!make_tmap_u8(&m[b], base, k, rows, 16u << b)) return false;
  return true;
}

}  // namespace

int mx_ffn_supported(int H, int I, int I_shared, int E) {
  if (H % 128 || I % 128 || I_shared % 128) return 0;
  // the compute shape is the fallback of every launch (mx_launch)
  return mx_smem_bytes<MxCompute>(E) <= XSMEM_LIMIT;
}

int launch_expert_ffn_mx(const FfnMxArgs& a, cudaStream_t s) {
  const int TK = a.T * a.topk;
  // without xq the shared expert is skipped: its segment gets no rows and
  // its maps and scales are set on the routed tensors (never read)
  const bool shared = a.xq != nullptr;
  const int Ts = shared ? a.T : 0;
  // ---- up projection + SwiGLU + power-of-two re-quantization
  MxParams up;
  std::memset(&up, 0, sizeof(up));
  bool ok =
      mx_token_maps(up.tok_routed, a.xpq, a.H, TK) &&
      (shared ? mx_token_maps(up.tok_shared, a.xq, a.H, a.T)
              : mx_token_maps(up.tok_shared, a.xpq, a.H, TK)) &&
      make_tmap_u8(&up.wa_routed, a.w1, a.H, (uint64_t)a.E * a.I, XM) &&
      make_tmap_u8(&up.wb_routed, a.w3, a.H, (uint64_t)a.E * a.I, XM) &&
      (shared ? make_tmap_u8(&up.wa_shared, a.ws1, a.H, a.I_shared, XM) &&
                    make_tmap_u8(&up.wb_shared, a.ws3, a.H, a.I_shared, XM)
              : make_tmap_u8(&up.wa_shared, a.w1, a.H,
                             (uint64_t)a.E * a.I, XM) &&
                    make_tmap_u8(&up.wb_shared, a.w3, a.H,
                                 (uint64_t)a.E * a.I, XM));
  if (!ok) return MOE_ERR_CUDA;
  up.ts_routed = a.xps;
  up.ts_shared = shared ? a.xs : a.xps;
  up.sa_routed = a.w1s;
  up.sb_routed = a.w3s;
  up.sa_shared = shared ? a.ws1s : a.w1s;
  up.sb_shared = shared ? a.ws3s : a.w3s;
  up.offsets = a.offsets;
  up.q_routed = a.mq;
  up.qs_routed = a.ms;
  up.q_shared = a.msq;
  up.qs_shared = a.mss;
  up.status = a.status;
  up.wait_limit_ns = a.wait_limit_ns;
  up.E = a.E;
  up.T = Ts;
  up.TK = TK;
  up.n_routed = a.I;
  up.n_shared = a.I_shared;
  up.k_routed = a.H;
  up.k_shared = a.H;
  int rc = mx_launch<kMxUp>(up, s);
  if (rc != MOE_OK) return rc;

  // ---- down projection
  MxParams dn;
  std::memset(&dn, 0, sizeof(dn));
  ok = mx_token_maps(dn.tok_routed, a.mq, a.I, TK) &&
       (shared ? mx_token_maps(dn.tok_shared, a.msq, a.I_shared, a.T)
               : mx_token_maps(dn.tok_shared, a.mq, a.I, TK)) &&
       make_tmap_u8(&dn.wa_routed, a.w2, a.I, (uint64_t)a.E * a.H, XM) &&
       (shared ? make_tmap_u8(&dn.wa_shared, a.ws2, a.I_shared, a.H, XM)
               : make_tmap_u8(&dn.wa_shared, a.w2, a.I, (uint64_t)a.E * a.H,
                              XM));
  if (!ok) return MOE_ERR_CUDA;
  dn.wb_routed = dn.wa_routed;
  dn.wb_shared = dn.wa_shared;
  dn.ts_routed = a.ms;
  dn.ts_shared = shared ? a.mss : a.ms;
  dn.sa_routed = a.w2s;
  dn.sb_routed = a.w2s;
  dn.sa_shared = shared ? a.ws2s : a.w2s;
  dn.sb_shared = shared ? a.ws2s : a.w2s;
  dn.offsets = a.offsets;
  dn.y_routed = a.yp;
  dn.y_shared = a.ys;
  dn.status = a.status;
  dn.wait_limit_ns = a.wait_limit_ns;
  dn.E = a.E;
  dn.T = Ts;
  dn.TK = TK;
  dn.n_routed = a.H;
  dn.n_shared = a.H;
  dn.k_routed = a.I;
  dn.k_shared = a.I_shared;
  return mx_launch<kMxDown>(dn, s);
}

}  // namespace moe
