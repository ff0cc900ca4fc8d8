// Host-side launch interface between the C-ABI layer (moe_api.cu) and the
// kernel files.  Every launcher validates nothing (the API layer did) and
// returns the cudaGetLastError() of its launches.
#pragma once

#include <cuda.h>

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

// Routing blocks (the per-block expert histogram and the stable dispatch
// order are both computed over them): consecutive token ranges of at most
// 64 tokens, each with one row of per-expert counts.  From 32 blocks
// on their number is rounded up to a multiple of the B300's 148 SMs, so
// every SM routes the same number of tokens (the work per token is fixed;
// 256 blocks of 64 tokens at T = 16384 left 108 SMs with two blocks and 40
// with one).  Block b covers [route_block_start(b), route_block_start(b+1)).
constexpr int kRouteTokensPerBlock = 64;
constexpr int kRouteSmMultiple = 148;

inline int route_blocks(int T) {
  const int nb = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  return nb >= 32 ? (nb + kRouteSmMultiple - 1) / kRouteSmMultiple *
                        kRouteSmMultiple
                  : nb;
}

__host__ __device__ inline int route_block_start(int b, int T, int nb) {
  return static_cast<int>(static_cast<long long>(b) * T / nb);
}

struct DevStatus;

// ---- routing.cu
// offset [E] may be NULL (no additive term)
cudaError_t launch_router_logits(const uint16_t* x, const float* w_router,
                                 const float* offset, float* logits, int T,
                                 int H, int E, cudaStream_t s);
cudaError_t launch_route(const float* logits, const float* bias, int T, int E,
                         int n_group, int topk_group, int topk,
                         int32_t* topk_idx, float* topk_gate,
                         int32_t* block_counts, cudaStream_t s);
cudaError_t launch_block_counts(const int32_t* topk_idx, int T, int E,
                                int topk, int32_t* block_counts,
                                DevStatus* st, cudaStream_t s);
// column scan of the per-block histograms: counts[e] (may be NULL),
// block_prefix[blk][e] = counts of e in blocks before blk (may be NULL),
// and -- if bias != nullptr -- the bias step on the final counts
cudaError_t launch_scan(const int32_t* block_counts, int T, int E, int topk,
                        int32_t* counts, int32_t* block_prefix, float* bias,
                        float gamma, cudaStream_t s);
// stable dispatch order from topk_idx, counts and block_prefix; writes
// offsets[E+1] and load_stats[3] when non-NULL
cudaError_t launch_dest(const int32_t* topk_idx, const int32_t* counts,
                        const int32_t* block_prefix, int T, int E, int topk,
                        int32_t* offsets, int32_t* dest, int32_t* src_row,
                        float* load_stats, DevStatus* st, cudaStream_t s);
cudaError_t launch_gather(const uint16_t* x, const int32_t* dest, int T, int H,
                          int topk, uint16_t* xp, cudaStream_t s);
cudaError_t launch_combine(const uint16_t* x, const uint16_t* ys,
                           const uint16_t* yp, const int32_t* dest,
                           const float* gate, int T, int H, int topk,
                           uint16_t* out, cudaStream_t s);
cudaError_t launch_bias_update(const int32_t* counts, float* bias,
                               float* load_stats, int T, int E, int topk,
                               float gamma, cudaStream_t s);
// sequence-wise balance loss: sp [T, E] fp32 and flags [T, E] u8 are
// scratch, part_P / part_c [n_seq, rs, E] the per-split partial sums (used
// when seq_balance_splits() > 1; n_seq * rs * E <= kBalPartialElems);
// P and counts [n_seq, E] and loss [n_seq] are written
// backward of routing to the logits (gates; balance loss), one warp per
// token; accumulate != 0 adds to dz instead of overwriting it
cudaError_t launch_route_backward(const float* logits, const int32_t* idx,
                                  const float* dgate, int T, int E, int K,
                                  int accumulate, float* dz, DevStatus* st,
                                  cudaStream_t s);
cudaError_t launch_seq_balance_backward(const float* logits, int T, int E,
                                        int K, int seq_len, float alpha,
                                        const int32_t* counts_seq,
                                        const float* dloss, int accumulate,
                                        float* dz, cudaStream_t s);
// both: the gates' term, then the balance term, in one pass
cudaError_t launch_route_balance_backward(
    const float* logits, const int32_t* idx, const float* dgate, int T,
    int E, int K, int seq_len, float alpha, const int32_t* counts_seq,
    const float* dloss, int accumulate, float* dz, DevStatus* st,
    cudaStream_t s);
constexpr int kBalSplitTarget = 148;  // split up to 2 x this many CTAs
constexpr long long kBalPartialElems = 2LL * kBalSplitTarget * 32;
int seq_balance_splits(int T, int E, int seq_len);
cudaError_t launch_seq_balance(const float* logits, int T, int E, int topk,
                               int seq_len, float alpha, float* sp,
                               uint8_t* flags, float* P, int32_t* counts,
                               float* part_P, int32_t* part_c, float* loss,
                               cudaStream_t s);

// ---- fp8.cu
// 1 x 128 tile quantization of x [R, C] bf16 (C % 128 == 0): codes to q
// [R, C] and scales to s [R, C/128] when q != NULL; with dest [R, K] != NULL
// also to the dispatch rows qp[dest[r*K+k]] / sp (bad rows: DEVICE_BOUNDS)
cudaError_t launch_quant_rows(const uint16_t* x, long long R, int C,
                              const int32_t* dest, int K, uint8_t* q,
                              float* s, uint8_t* qp, float* sp,
                              DevStatus* st, cudaStream_t stream);
// 128 x 128 block quantization of w [R, C] bf16 (both multiples of 128):
// codes q [R, C], scales s [R/128, C/128]
cudaError_t launch_quant_blocks(const uint16_t* w, long long R, int C,
                                uint8_t* q, float* s, cudaStream_t stream);
// the same with power-of-two scales, stored as UE8M0 bytes (e + 127)
cudaError_t launch_quant_rows_e8(const uint16_t* x, long long R, int C,
                                 const int32_t* dest, int K, uint8_t* q,
                                 uint8_t* s, uint8_t* qp, uint8_t* sp,
                                 DevStatus* st, cudaStream_t stream);
cudaError_t launch_quant_blocks_e8(const uint16_t* w, long long R, int C,
                                   uint8_t* q, uint8_t* s,
                                   cudaStream_t stream);

// ---- grouped_gemm.cu
struct FfnArgs {
  int T, H, E, topk, I, I_shared;
  const uint16_t *xp, *x;          // A of the up GEMM
  // with xp == NULL: the routed rows are gathered from x inside the up
  // GEMM, row r being token src_row[r] / topk (moe_permute's src_row)
  const int32_t* src_row = nullptr;
  const int32_t* offsets;          // [E+1]
  const uint16_t *w1, *w3, *w2;    // routed weights
  const uint16_t *ws1, *ws3, *ws2; // shared expert
  uint16_t *h, *hs;                // intermediate [T*K, I], [T, I_shared]
  uint16_t *yp, *ys;               // outputs
  DevStatus* status;
  uint64_t wait_limit_ns;
  void* between_event = nullptr;   // cudaEvent_t recorded between the GEMMs
};
// 0 on success, else a moe_status_t (encoding or launch failure)
int launch_expert_ffn(const FfnArgs& a, cudaStream_t s);

// ---- expert_backward.cu
struct BwdArgs {
  int T, H, E, topk, I, I_shared;
  const uint16_t *x, *dout;                 // [T, H]
  const int32_t *topk_idx, *dest, *offsets, *counts;  // unpadded dispatch
  const float* gate;                         // [T, K]
  const uint16_t *w1, *w3, *w2, *ws1, *ws3, *ws2;
  int32_t *poff, *pdest;                     // [E+1], [T*K]
  int* ticket;                               // [1] weight-gradient tasks
  float* gp;                                 // [cap]
  uint16_t *xpp, *dpp;                       // [cap, H]
  float *p_r, *q_r;                          // [cap, I]
  uint16_t *hg_r, *dp_r, *dq_r;              // [cap, I]
  float* dgp;                                // [cap, ceil(I / 256)]
  uint16_t* dxpp;                            // [cap, H]
  float *p_s, *q_s;                          // [T, I_s]
  uint16_t *hg_s, *dp_s, *dq_s;              // [T, I_s]
  uint16_t* dxs;                             // [T, H]
  uint16_t* dx;                              // [T, H] out
  float* dgate;                              // [T, K] out
  float *dw1, *dw3, *dw2, *dws1, *dws3, *dws2;  // out (fp32)
  int accumulate;
  DevStatus* status;
  uint64_t wait_limit_ns;
  // cudaEvent_t handles recorded before each of the 6 stages and after the
  // last (dispatch, recompute, dgrad down, dgrad up, wgrad, finalize), or
  // NULL
  void* const* events = nullptr;
};
// rows of the padded dispatch: T*K + 15*E (each segment rounded up to 16)
size_t expert_backward_rows_cap(int T, int K, int E);
int launch_expert_backward(const BwdArgs& a, cudaStream_t s);

// ---- ep.cu
int ep_plan_max_cells();  // n_src * n_local limit of launch_ep_plan
cudaError_t launch_ep_plan(const int32_t* counts, int n_src, int n_local,
                           long long rows, int32_t* perm,
                           int32_t* offsets_local, DevStatus* st,
                           cudaStream_t s);
cudaError_t launch_ep_rows(const void* in, long long rows,
                           long long row_bytes, const int32_t* perm,
                           int inverse, void* out, DevStatus* st,
                           cudaStream_t s);

// ---- fp8_gemm.cu
struct FfnFp8Args {
  int T, H, E, topk, I, I_shared;
  const uint8_t *xpq, *xq;         // E4M3 token rows [T*K, H], [T, H]
  const float *xps, *xs;           // their 1 x 128 scales
  const int32_t* offsets;          // [E+1]
  const uint8_t *w1, *w3, *w2;     // routed weights, E4M3
  const float *w1s, *w3s, *w2s;    // their 128 x 128 block scales
  const uint8_t *ws1, *ws3, *ws2;  // shared expert
  const float *ws1s, *ws3s, *ws2s;
  uint8_t *mq, *msq;               // intermediate codes [T*K, I], [T, I_s]
  float *ms, *mss;                 // their scales
  uint16_t *yp, *ys;               // outputs, bf16
  DevStatus* status;
  uint64_t wait_limit_ns;
};
// 1 when the FP8 kernels have a shape for these sizes
int fp8_ffn_supported(int H, int I, int I_shared, int E);
int launch_expert_ffn_fp8(const FfnFp8Args& a, cudaStream_t s);

// ---- mx_gemm.cu
// The FP8 expert FFNs with power-of-two (UE8M0) group scales applied by
// the tensor cores' block scaling; same tensors as FfnFp8Args, scales as
// UE8M0 bytes (2^(b - 127)).
struct FfnMxArgs {
  int T, H, E, topk, I, I_shared;
  const uint8_t *xpq, *xq;         // E4M3 token rows [T*K, H], [T, H]
  const uint8_t *xps, *xs;         // their 1 x 128 scales (UE8M0)
  const int32_t* offsets;          // [E+1]
  const uint8_t *w1, *w3, *w2;     // routed weights, E4M3
  const uint8_t *w1s, *w3s, *w2s;  // their 128 x 128 block scales (UE8M0)
  const uint8_t *ws1, *ws3, *ws2;  // shared expert
  const uint8_t *ws1s, *ws3s, *ws2s;
  uint8_t *mq, *msq;               // intermediate codes [T*K, I], [T, I_s]
  uint8_t *ms, *mss;               // their scales (UE8M0)
  uint16_t *yp, *ys;               // outputs, bf16
  DevStatus* status;
  uint64_t wait_limit_ns;
};
int mx_ffn_supported(int H, int I, int I_shared, int E);
int launch_expert_ffn_mx(const FfnMxArgs& a, cudaStream_t s);

// ---- router_gemm.cu
// router logits on the tensor cores from the exact 3-way bf16 split of the
// fp32 router weight (w_split [3, E, H], see launch_split_router_weight);
// returns MOE_ERR_UNSUPPORTED when E is not a multiple of 16
// (partial: [router_ksplit(T,H,E), T, E] fp32 scratch, used when the
// reduction over H is split; may be NULL when router_ksplit() == 1)
int launch_router_logits_tc(const uint16_t* x, const uint16_t* w_split,
                            const float* offset, float* logits,
                            float* partial, int T, int H, int E,
                            DevStatus* status, uint64_t wait_limit_ns,
                            cudaStream_t s);
int router_tile_n(int T, int E);  // 0: the tensor-core path does not apply
int router_ksplit(int T, int H, int E);  // k ranges of the router GEMM
// (routing.cu) the exact split itself
cudaError_t launch_split_router_weight(const float* w, int E, int H,
                                       uint16_t* w_split, cudaStream_t s);

// ---- host_util.cu
// 2-D bf16 row-major [outer, inner] tensor map, box [box_outer rows, 64
// elements], 128-byte swizzle; false if encoding fails
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner,
                    uint64_t outer, uint32_t box_outer);
// the same for a byte tensor (E4M3 codes): box [box_outer rows, 128 B]
bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t inner,
                  uint64_t outer, uint32_t box_outer);
// 3-D fp32 tensor [mats][rows][n] (n contiguous) for TMA stores and
// reductions of 32 x 32 tiles, 128-byte swizzle
bool make_tmap_f32_3d_store(CUtensorMap* m, void* base, uint64_t n,
                            uint64_t rows, uint64_t mats);
int sm_count();
int gemm_ctas();           // persistent CTAs of the expert GEMMs
void set_gemm_ctas(int n); // 0: one per SM

}  // namespace moe
