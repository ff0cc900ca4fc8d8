// Grouped BF16 GEMMs of the expert FFNs on the sm_103a tensor cores.
//
// Every routed expert of the DeepSeek-V3 MoE layer is a SwiGLU FFN with
// three matrices ("02 · DeepSeek-V3" (PaperTrace) §1.1); the shared expert
// has the same form and runs on every token (§1.1; §5.1 treats it as a
// ninth, always-chosen expert).  Rows of the dispatched activations are
// grouped by expert (segments [offsets[e], offsets[e+1])), plus one segment
// for the shared expert over all T tokens:
//
//   up   (MODE kUp):   h = silu(A W1^T) * (A W3^T)   A = xp rows | x rows
//   down (MODE kDown): y = h W2^T
//
// Weights are the MMA's M side and tokens its N side ("swap AB"): a unit
// computes D[f, t] = W[f, :] . A[t, :] for 2 x 128 weight rows f and one
// chunk of N <= 256 token rows t of one segment.  N is the chunk's row
// count rounded up to 16 and is set per unit in the instruction descriptor,
// so a segment of 140 rows costs 144 columns of MMA work, not two 128-row
// tiles; segments longer than 256 rows are cut into equal chunks.  The two
// weight tiles of a unit feed two accumulators:
//   up:   W1 rows [f0, f0+128) and W3 rows [f0, f0+128) -- gate and up value
//         of feature f land in the same TMEM lane, so SwiGLU needs no
//         exchange between threads
//   down: W2 rows [f0, f0+128) and [f0+128, f0+256)
//
// Design (one persistent CTA per SM, 7 warps):
//   warp 0 lane 0   weight producer: the two 128x64 weight tiles of every
//                   k-block into a deep ring (the HBM stream: its depth is
//                   what keeps enough bytes in flight per SM)
//   warp 2 lane 0   token producer: the Nx64 token tile (boxes of
//                   128/64/32/16 rows summing to N) into a shallow ring (the
//                   rows are L2-resident, re-read by every feature block)
//                   both with 128-byte swizzle and mbarrier completion.  In
//                   the gather mode of the up projection the routed rows
//                   are not copied out beforehand: the warp reads the
//                   chunk's token ids (dispatch order / top-K) once per
//                   unit and every k-block gathers the rows from x itself,
//                   four rows per TMA gather4
//   warp 1 lane 0   tcgen05.mma issuer (M=128, N per unit, K=16), fp32
//                   accumulators in tensor memory; warp 1 owns the TMEM
//                   allocation (512 columns = two slots of 256)
//   warps 3..6      epilogue: tcgen05.ld, SwiGLU (up) or conversion (down),
//                   bf16 stores of the valid rows and features
// TMEM: a unit with N <= 128 puts both accumulators in one 256-column slot,
// so consecutive such units alternate slots and the epilogue of one overlaps
// the MMAs of the next; a unit with N > 128 takes both slots.
// The unit list -- the shared segment first (its units are the longest),
// then the routed experts, each as (feature block, chunk) with the chunk
// fastest so CTAs sharing a weight tile run side by side and hit L2 -- is
// derived on the device from `offsets`; nothing is read back to the host.
//
// Every wait is bounded (MOE_ERR_TIMEOUT in the status word, then a clean
// exit: in-flight copies and MMAs are drained, TMEM is freed).
#include <cuda.h>

#include <cstdint>
#include <cstring>

#include "device_common.cuh"
#include "internal.h"
#include "unit_list.cuh"

namespace moe {
namespace {

constexpr int BM = 128;         // weight rows per accumulator = MMA M
constexpr int BK = 64;          // K per stage: 64 bf16 = one 128 B row
constexpr int UMMA_K = 16;      // K of one kind::f16 MMA
// Two pipeline shapes, chosen per launch from the mean rows per routed
// expert (T*K/E): below the bf16 ridge of ~256 rows (FLOP per weight byte
// ~= rows) the GEMM streams weights from HBM and wants short token chunks
// with a deeper token ring; above it, it is tensor-bound and wants the
// widest MMA (N = 256).  Both were measured best of a sweep on B300.
//   NT  largest token chunk = largest MMA N (<= 256, multiple of 16)
//   WS  depth of the weight ring (the HBM stream)
//   TS  depth of the token ring (L2-resident rows, re-read per block)
template <int NT_, int WS_, int TS_>
struct Pipe {
  static constexpr int NT = NT_;
  static constexpr int WS = WS_;
  static constexpr int TS = TS_;
};
using PipeStream = Pipe<192, 4, 3>;   // mean rows per expert < 256
using PipeCompute = Pipe<256, 4, 2>;  // mean rows per expert >= 256
constexpr int kComputeRows = 256;
constexpr int kEpiWarps = 4;  // one per TMEM lane quadrant
constexpr int kEpiWarp0 = 3;  // warps 0..2: weight producer, MMA, token producer
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int SLOT = 256;       // TMEM columns per accumulator slot
constexpr int kTokBoxes = 4;    // token boxes of 16, 32, 64, 128 rows
constexpr uint32_t W_BYTES = BM * BK * 2;         // one weight tile
constexpr uint32_t WSTAGE_BYTES = 2 * W_BYTES;    // both weight tiles
constexpr uint32_t TMEM_COLS = 2 * SLOT;          // two slots
constexpr size_t kSmemLimit = 232448;             // 227 KB per CTA

// shared-memory layout of one pipeline shape
template <class P>
struct Ring {
  static constexpr uint32_t TSTAGE_BYTES = P::NT * BK * 2;  // token tile
  static constexpr uint32_t BYTES =
      P::WS * WSTAGE_BYTES + P::TS * TSTAGE_BYTES;
  static constexpr int BARS = 2 * P::WS + 2 * P::TS + 5;
  static_assert(P::NT % 16 == 0 && P::NT >= 16 && P::NT <= SLOT, "chunk");
  static_assert(TSTAGE_BYTES % 1024 == 0, "swizzle atoms stay aligned");
};
constexpr uint64_t kDrainNs = 2000000000ull;

enum { kUp = 0, kDown = 1 };
enum {
  kSiteProducer = 21,
  kSiteMmaAcc = 22,
  kSiteMmaFull = 23,
  kSiteEpilogue = 24,
  kSiteDrain = 25,
  kSiteOffsets = 26
};

struct GemmParams {  // CUtensorMap members carry their 64-byte alignment
  CUtensorMap tok_routed[kTokBoxes];  // up: xp [TK, H]   down: h  [TK, I]
  CUtensorMap tok_shared[kTokBoxes];  // up: x  [T, H]    down: hs [T, I_s]
  CUtensorMap wa_routed;  // up: w1 [E*I, H]     down: w2 [E*H, I]
  CUtensorMap wb_routed;  // up: w3 [E*I, H]     down: w2 (rows + 128)
  CUtensorMap wa_shared;  // up: ws1 [I_s, H]    down: ws2 [H, I_s]
  CUtensorMap wb_shared;  // up: ws3 [I_s, H]    down: ws2 (rows + 128)
  CUtensorMap tok_gather; // gather mode: x [T, H], boxes of one row
  const int32_t* src_row; // gather mode: [TK] t * topk + k of each row
  int topk, gather;       // gather: routed rows gathered from x
  const int32_t* offsets; // [E+1]
  uint16_t* out_routed;   // up: h [TK, I]       down: yp [TK, H]
  uint16_t* out_shared;   // up: hs [T, I_s]     down: ys [T, H]
  DevStatus* status;
  unsigned long long wait_limit_ns;
  int E, T, TK;
  int n_routed, n_shared;  // output features of a routed / the shared segment
  int k_routed, k_shared;  // reduction length of a routed / the shared one
};

// output features one unit produces
template <int MODE>
struct Feat {
  static constexpr int FB = (MODE == kUp) ? BM : 2 * BM;
};

template <int MODE, class P>
__global__ void __launch_bounds__(kThreads, 1)
    expert_gemm_kernel(const __grid_constant__ GemmParams p) {
  constexpr int FB = Feat<MODE>::FB;
  constexpr int NT = P::NT, kWStages = P::WS, kTStages = P::TS;
  constexpr uint32_t TSTAGE_BYTES = Ring<P>::TSTAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;                                  // weight ring
  uint8_t* sT = smem + kWStages * WSTAGE_BYTES;        // token ring
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ring<P>::BYTES);
  uint64_t* wfull = bars;
  uint64_t* wempty = wfull + kWStages;
  uint64_t* kfull = wempty + kWStages;
  uint64_t* kempty = kfull + kTStages;
  uint64_t* tfull = kempty + kTStages;  // per TMEM slot
  uint64_t* tempty = tfull + 2;         // per TMEM slot
  uint64_t* drain = tempty + 2;
  volatile uint32_t* misc =
      reinterpret_cast<volatile uint32_t*>(bars + Ring<P>::BARS);
  // misc[0] TMEM base, misc[1] abort flag, misc[2] bad-offsets flag
  const int E = p.E;
  const int NS = E + 1;  // the shared segment (0) + the routed ones
  int* useg = reinterpret_cast<int*>(const_cast<uint32_t*>(misc) + 4);
  int* srows = useg + NS + 1;
  int* srow0 = srows + NS;
  // gather mode: the current chunk's token ids (16-byte aligned)
  int* s_tok = reinterpret_cast<int*>(
      (reinterpret_cast<uintptr_t>(srow0 + NS) + 15) & ~uintptr_t(15));

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
      mbar_init(smem_u32(&tempty[i]), 32 * kEpiWarps);
    }
    mbar_init(smem_u32(drain), 1);
    misc[1] = 0;
    misc[2] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
#pragma unroll
    for (int b = 0; b < kTokBoxes; ++b) {
      prefetch_tmap(&p.tok_routed[b]);
      prefetch_tmap(&p.tok_shared[b]);
    }
    prefetch_tmap(&p.wa_routed);
    prefetch_tmap(&p.wb_routed);
    prefetch_tmap(&p.wa_shared);
    prefetch_tmap(&p.wb_shared);
    if (p.gather) prefetch_tmap(&p.tok_gather);
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
      // ----------------------------------------------- weight producer
      uint32_t stage = 0, phase = 0, issued = 0;
      const uint64_t pol_w = policy_evict_first();
      // weight tiles of unit u: maps, first rows, k-blocks
      auto unit_w = [&](int u, const CUtensorMap*& wa, const CUtensorMap*& wb,
                        int& wrow, int& wrow_b) {
        const Unit w = decode_unit<NT>(u, useg, srow0, srows, NS);
        const bool sh = (w.seg == 0);
        wa = sh ? &p.wa_shared : &p.wa_routed;
        wb = sh ? &p.wb_shared : &p.wb_routed;
        wrow = (sh ? 0 : (w.seg - 1) * p.n_routed) + w.f * FB;
        wrow_b = (MODE == kUp) ? wrow : wrow + BM;
        return (sh ? p.k_shared : p.k_routed) / BK;
      };
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const CUtensorMap *wa, *wb;
        int wrow, wrow_b;
        const int nkb = unit_w(u, wa, wb, wrow, wrow_b);
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
          tma_load_2d_hint(smem_u32(st), wa, kb * BK, wrow, fb, pol_w);
          tma_load_2d_hint(smem_u32(st + W_BYTES), wb, kb * BK, wrow_b, fb,
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
                          (i / kWStages) & 1, nullptr, kDrainNs, p.status,
                          kSiteDrain);
    }
    __syncwarp();
  } else if (warp == 2) {
    // -------------------------------------------------- token producer
    uint32_t stage = 0, phase = 0, issued = 0;
    const uint64_t pol_t = policy_evict_last();
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const Unit w = decode_unit<NT>(u, useg, srow0, srows, NS);
      const bool sh = (w.seg == 0);
      const bool gat = !sh && p.gather;
      const CUtensorMap* tok = sh ? p.tok_shared : p.tok_routed;
      const int nkb = (sh ? p.k_shared : p.k_routed) / BK;
      const uint32_t tx = (uint32_t)w.n * BK * 2;
      if (gat) {
        // the token of every row of the chunk; the padding rows up to the
        // MMA's N repeat the last one (their columns are not stored)
        for (int i = lane; i < w.n; i += 32)
          s_tok[i] = p.src_row[w.row0 + min(i, w.rows - 1)] / p.topk;
        __syncwarp();
      }
      int ok = 1;
      for (int kb = 0; kb < nkb; ++kb) {
        if (lane == 0) {
          ok = mbar_wait_bounded(smem_u32(&kempty[stage]), phase ^ 1,
                                 abort_flag, limit, p.status, kSiteProducer);
          if (ok) {
            const uint32_t fb = smem_u32(&kfull[stage]);
            uint8_t* stok = sT + stage * TSTAGE_BYTES;
            mbar_arrive_expect_tx(fb, tx);
            if (gat) {
              for (int g = 0; g < w.n; g += 4)
                tma_gather4(smem_u32(stok + g * BK * 2), &p.tok_gather,
                            kb * BK, *reinterpret_cast<const int4*>(s_tok + g),
                            fb);
            } else if (w.n == 256) {
              // token rows [row0, row0 + n) as boxes of 128/64/32/16 rows
              tma_load_2d_hint(smem_u32(stok), &tok[3], kb * BK, w.row0, fb,
                               pol_t);
              tma_load_2d_hint(smem_u32(stok + 128 * BK * 2), &tok[3],
                               kb * BK, w.row0 + 128, fb, pol_t);
            } else {
              int off = 0;
#pragma unroll
              for (int b = kTokBoxes - 1; b >= 0; --b) {
                if ((w.n >> 4) & (1 << b)) {
                  tma_load_2d_hint(smem_u32(stok + off * BK * 2), &tok[b],
                                   kb * BK, w.row0 + off, fb, pol_t);
                  off += 16 << b;
                }
              }
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++issued;
        if (++stage == kTStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      __syncwarp();  // s_tok is rewritten for the next unit
      if (!ok) break;
    }
    if (lane == 0) {
      const uint32_t first = issued > kTStages ? issued - kTStages : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait_bounded(smem_u32(&kfull[i % kTStages]),
                          (i / kTStages) & 1, nullptr, kDrainNs, p.status,
                          kSiteDrain);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------- MMA
      uint32_t wstage = 0, wphase = 0, kstage = 0, kphase = 0;
      uint32_t tph = 0;  // bit s: parity of the uses of TMEM slot s so far
      int slot = 0;
      bool any = false;
      for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const Unit w = decode_unit<NT>(u, useg, srow0, srows, NS);
        const int nkb = ((w.seg == 0) ? p.k_shared : p.k_routed) / BK;
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
        const uint32_t idesc = idesc_bf16_f32(BM, w.n);
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
            tc_mma_f16(da, sw128_kmajor_desc(s0 + kk * UMMA_K * 2), bdesc,
                       idesc, acc);
            tc_mma_f16(db, sw128_kmajor_desc(s0 + W_BYTES + kk * UMMA_K * 2),
                       bdesc, idesc, acc);
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
        mbar_wait_bounded(smem_u32(drain), 0, nullptr, kDrainNs, p.status,
                          kSiteDrain);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- epilogue
    // Every accumulator column of a unit is read into registers (bf16
    // pairs) before any global store, so TMEM goes back to the MMA warp as
    // soon as it is read and the slow, scattered stores overlap the next
    // unit's MMAs instead of delaying them.
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r = q * 32 + lane;
    uint32_t tph = 0;  // bit s: parity of the uses of TMEM slot s so far
    int slot = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      const Unit w = decode_unit<NT>(u, useg, srow0, srows, NS);
      const bool wide = w.n > SLOT / 2;
      const int s1 = wide ? (slot ^ 1) : slot;
      int ok = 0;
      if (lane == 0) {
        ok = mbar_wait_bounded(smem_u32(&tfull[slot]), (tph >> slot) & 1,
                               abort_flag, limit, p.status, kSiteEpilogue);
        if (ok && wide)
          ok = mbar_wait_bounded(smem_u32(&tfull[s1]), (tph >> s1) & 1,
                                 abort_flag, limit, p.status, kSiteEpilogue);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
      const uint32_t ta = tmem_base + lane_off + slot * SLOT;
      const uint32_t tb =
          wide ? tmem_base + lane_off + s1 * SLOT : ta + SLOT / 2;
      const bool sh = (w.seg == 0);
      uint16_t* out = sh ? p.out_shared : p.out_routed;
      const int ld = sh ? p.n_shared : p.n_routed;
      // feature columns of this thread's TMEM lane in both accumulators
      const int fa = w.f * FB + r;
      const int fbc = (MODE == kUp) ? fa : fa + BM;
      uint16_t* obase = out + (size_t)w.row0 * ld;
      auto release = [&](int sl) {
        tc_fence_before();
        mbar_arrive(smem_u32(&tempty[sl]));
      };
      if (MODE == kUp) {
        uint32_t pk[NT / 2];
#pragma unroll
        for (int c = 0; c < NT / 16; ++c) {
          if (16 * c < w.n) {
            uint32_t a[16], b[16];
            tmem_ld16(ta + 16 * c, a);
            tmem_ld16(tb + 16 * c, b);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              pk[8 * c + i] = pack_bf16x2(
                  silu_f(__uint_as_float(a[2 * i])) *
                      __uint_as_float(b[2 * i]),
                  silu_f(__uint_as_float(a[2 * i + 1])) *
                      __uint_as_float(b[2 * i + 1]));
          }
        }
        release(slot);
        if (wide) release(s1);
        if (fa < ld) store_packed<NT>(pk, obase + fa, ld, w.rows);
      } else {
        // a wide unit's accumulators sit in two slots: each is released as
        // soon as it is read; a narrow unit's slot after both are read
        uint32_t pk[NT / 2];
        load_packed<NT>(ta, w.n, pk);
        if (wide) release(slot);
        if (fa < ld) store_packed<NT>(pk, obase + fa, ld, w.rows);
        load_packed<NT>(tb, w.n, pk);
        release(s1);
        if (fbc < ld) store_packed<NT>(pk, obase + fbc, ld, w.rows);
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
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <class P>
size_t smem_bytes(int E) {
  return 1024 + Ring<P>::BYTES + Ring<P>::BARS * sizeof(uint64_t) +
         4 * sizeof(uint32_t) + sizeof(int) * (3 * (E + 1) + 1) + 16 +
         sizeof(int) * P::NT;
}

template <int MODE, class P>
int launch_shape(const GemmParams& gp, cudaStream_t s) {
  auto kern = expert_gemm_kernel<MODE, P>;
  const size_t smem = smem_bytes<P>(gp.E);
  if (smem > kSmemLimit) return MOE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MOE_ERR_CUDA;
  kern<<<gemm_ctas(), kThreads, smem, s>>>(gp);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// the pipeline shape for this launch's mean rows per routed expert
template <int MODE>
int launch_one(const GemmParams& gp, cudaStream_t s) {
  const long long mean_rows = gp.E > 0 ? (long long)gp.TK / gp.E : 0;
  return mean_rows >= kComputeRows ? launch_shape<MODE, PipeCompute>(gp, s)
                                   : launch_shape<MODE, PipeStream>(gp, s);
}

// token-operand maps of one [rows, k] bf16 tensor, boxes of 16..128 rows
bool token_maps(CUtensorMap (&m)[kTokBoxes], const void* base, uint64_t k,
                uint64_t rows) {
  for (int b = 0; b < kTokBoxes; ++b)
    if (!make_tmap_bf16(&m[b], base, k, rows, 16u << b)) return false;
  return true;
}

}  // namespace

int launch_expert_ffn(const FfnArgs& a, cudaStream_t s) {
  const int TK = a.T * a.topk;
  // without x the shared expert is skipped: its segment gets no rows and
  // its maps are encoded on the routed tensors (never read)
  const bool shared = a.x != nullptr;
  const int Ts = shared ? a.T : 0;
  // without xp the routed rows are gathered from x by src_row
  const bool gather = a.xp == nullptr;
  if (gather && (a.x == nullptr || a.src_row == nullptr))
    return MOE_ERR_INVALID_ARG;
  // ---- up projection + SwiGLU
  GemmParams up;
  std::memset(&up, 0, sizeof(up));
  bool ok = token_maps(up.tok_routed, gather ? a.x : a.xp, a.H,
                       gather ? a.T : TK) &&
            make_tmap_bf16(&up.tok_gather, shared ? a.x : a.xp, a.H,
                           shared ? a.T : TK, 1) &&
            (shared ? token_maps(up.tok_shared, a.x, a.H, a.T)
                    : token_maps(up.tok_shared, a.xp, a.H, TK)) &&
            make_tmap_bf16(&up.wa_routed, a.w1, a.H, (uint64_t)a.E * a.I, BM) &&
            make_tmap_bf16(&up.wb_routed, a.w3, a.H, (uint64_t)a.E * a.I, BM) &&
            (shared ? make_tmap_bf16(&up.wa_shared, a.ws1, a.H, a.I_shared, BM) &&
                          make_tmap_bf16(&up.wb_shared, a.ws3, a.H, a.I_shared, BM)
                    : make_tmap_bf16(&up.wa_shared, a.w1, a.H,
                                     (uint64_t)a.E * a.I, BM) &&
                          make_tmap_bf16(&up.wb_shared, a.w3, a.H,
                                         (uint64_t)a.E * a.I, BM));
  if (!ok) return MOE_ERR_CUDA;
  up.gather = gather ? 1 : 0;
  up.src_row = a.src_row;
  up.topk = a.topk;
  up.offsets = a.offsets;
  up.out_routed = a.h;
  up.out_shared = a.hs;
  up.status = a.status;
  up.wait_limit_ns = a.wait_limit_ns;
  up.E = a.E;
  up.T = Ts;
  up.TK = TK;
  up.n_routed = a.I;
  up.n_shared = a.I_shared;
  up.k_routed = a.H;
  up.k_shared = a.H;
  int rc = launch_one<kUp>(up, s);
  if (rc != MOE_OK) return rc;
  if (a.between_event != nullptr)
    cudaEventRecord(static_cast<cudaEvent_t>(a.between_event), s);

  // ---- down projection
  GemmParams dn;
  std::memset(&dn, 0, sizeof(dn));
  ok = token_maps(dn.tok_routed, a.h, a.I, TK) &&
       (shared ? token_maps(dn.tok_shared, a.hs, a.I_shared, a.T)
               : token_maps(dn.tok_shared, a.h, a.I, TK)) &&
       make_tmap_bf16(&dn.wa_routed, a.w2, a.I, (uint64_t)a.E * a.H, BM) &&
       (shared ? make_tmap_bf16(&dn.wa_shared, a.ws2, a.I_shared, a.H, BM)
               : make_tmap_bf16(&dn.wa_shared, a.w2, a.I,
                                (uint64_t)a.E * a.H, BM));
  if (!ok) return MOE_ERR_CUDA;
  dn.wb_routed = dn.wa_routed;
  dn.wb_shared = dn.wa_shared;
  dn.offsets = a.offsets;
  dn.out_routed = a.yp;
  dn.out_shared = a.ys;
  dn.status = a.status;
  dn.wait_limit_ns = a.wait_limit_ns;
  dn.E = a.E;
  dn.T = Ts;
  dn.TK = TK;
  dn.n_routed = a.H;
  dn.n_shared = a.H;
  dn.k_routed = a.I;
  dn.k_shared = a.I_shared;
  return launch_one<kDown>(dn, s);
}

}  // namespace moe
