/*
 * moe.h -- C ABI of the B300 (sm_103a) DeepSeekMoE layer forward.
 *
 * The layer (DeepSeek-V3 MoE block, as described on "02 · DeepSeek-V3"
 * (PaperTrace) §1.1, §1.3 and §1.4):
 *
 *   s_{t,e}  = sigmoid(z_{t,e}),  z = x W_r^T              (eq. 15)
 *   u_{t,e}  = s_{t,e} + b_e      -- used for selection only (eq. 16)
 *   group score S_g = sum of the 2 largest u in group g; keep the best
 *   topk_group groups; choose the topk experts with the largest u among them
 *   g_{t,k}  = s_{t,e_k} / sum_j s_{t,e_j}                  (eq. 13)
 *   out_t    = x_t + FFN_shared(x_t) + sum_k g_{t,k} FFN_{e_k}(x_t)  (eq. 12)
 *   FFN(a)   = W2 (silu(W1 a) * (W3 a))                    (SwiGLU, §1.1)
 *   end of step: c_e = load of expert e over the batch; b_e -= gamma if
 *   c_e > T*K/E, b_e += gamma if c_e < T*K/E                (§1.4)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller, dense,
 *    row-major, 16-byte aligned (MOE_ERR_ALIGNMENT otherwise).  The library
 *    never allocates or frees device memory; scratch comes from a caller
 *    workspace sized by moe_workspace_bytes().
 *  - bf16 tensors are passed as uint16_t bit patterns.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream): no host synchronisation, no device-to-host copy.
 *  - Arguments are validated on the host before anything is launched;
 *    MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_ALIGNMENT /
 *    MOE_ERR_WORKSPACE are returned without touching the device.
 *    Launch failures return MOE_ERR_CUDA (checked with cudaGetLastError,
 *    without a sync).
 *  - Kernels that wait on asynchronous copies bound every wait; a wait that
 *    runs out records MOE_ERR_TIMEOUT in the workspace error word and the
 *    kernel returns cleanly.  moe_get_device_error() reports it.
 *  - Results are deterministic: no floating-point atomics, fixed orders.
 *  - T = 0 is valid: token-sized tensors may then be NULL; counts and
 *    offsets are zeroed, nothing else is written.
 *
 * Supported shapes (MOE_ERR_UNSUPPORTED outside them):
 *    H, I, I_shared: multiples of 64, >= 64
 *    E <= 32, or E in {64, 128, 256, 512, 1024}; E % n_group == 0;
 *    group size E/n_group >= 2; with L = max(1, E/32) experts per lane,
 *    (E/n_group) % L == 0 and (E/n_group)/L a power of two;
 *    1 <= topk_group <= n_group <= 32; 1 <= topk <= min(32,
 *    topk_group*E/n_group); T*(topk+1) < 2^31.
 */
#ifndef DEEPSEEKMOE_B300_MOE_H
#define DEEPSEEKMOE_B300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 4

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* NULL pointer, negative or inconsistent dims */
  MOE_ERR_UNSUPPORTED = 2,   /* valid dims the library has no kernel for    */
  MOE_ERR_ALIGNMENT = 3,     /* a pointer is not 16-byte aligned            */
  MOE_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than required     */
  MOE_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed           */
  MOE_ERR_TIMEOUT = 6,       /* a bounded device-side wait ran out          */
  MOE_ERR_DEVICE_BOUNDS = 7  /* a device-side index check failed            */
} moe_status_t;

/* A cudaStream_t, passed as an opaque handle so this header needs no CUDA
 * include.  NULL selects the legacy default stream. */
typedef void* moe_stream_t;

/* Layer dimensions.  Names follow the pages: T tokens, H hidden size, E
 * routed experts, n_group expert groups ("nodes" on the pages), topk_group
 * groups kept per token (4 for V3), topk experts per token (8 for V3), I the
 * routed expert intermediate size (2048 for V3), I_shared the shared expert
 * intermediate size, gamma the bias step (0.001 for V3). */
typedef struct {
  int32_t T;
  int32_t H;
  int32_t E;
  int32_t n_group;
  int32_t topk_group;
  int32_t topk;
  int32_t I;
  int32_t I_shared;
  float gamma;
} moe_dims_t;

/* Expert and router weights (device pointers, caller-owned, read only).
 *   w_router [E, H]    fp32   router vectors, one row per expert
 *   router_offset [E]  fp32   optional (NULL = none) additive term of the
 *                             router's linear map, z = x W_r^T + o.  V3's
 *                             router has none; a benchmark can put a
 *                             per-expert preference there to skew the load.
 *   w1       [E, I, H] bf16   gate projection of each routed expert
 *   w3       [E, I, H] bf16   up projection
 *   w2       [E, H, I] bf16   down projection
 *   ws1 [I_shared, H], ws3 [I_shared, H], ws2 [H, I_shared]: shared expert
 *   router_split [3, E, H] bf16  optional (NULL = none): the exact bf16
 *                             split of w_router that moe_router_weight_split
 *                             wrote; with it moe_forward does not split the
 *                             router weight again on every call.  It must
 *                             be the split of this w_router (not checked).
 */
typedef struct {
  const float* w_router;
  const uint16_t* w1;
  const uint16_t* w3;
  const uint16_t* w2;
  const uint16_t* ws1;
  const uint16_t* ws3;
  const uint16_t* ws2;
  const float* router_offset;
  const uint16_t* router_split;
} moe_weights_t;

/* Which entry point a workspace is sized for. */
typedef enum {
  MOE_WS_ROUTE = 0,
  MOE_WS_PERMUTE = 1,
  MOE_WS_EXPERT_FFN = 2,
  MOE_WS_FORWARD = 3,
  MOE_WS_ROUTER_LOGITS = 4,
  MOE_WS_SEQ_BALANCE = 5,
  MOE_WS_EXPERT_FFN_FP8 = 6,
  MOE_WS_EXPERT_BWD = 7,
  MOE_WS_EXPERT_FFN_MX = 8
} moe_ws_kind_t;

/* Bytes of device workspace `which` needs for dims `d` (0 if d is invalid).
 * A MOE_WS_FORWARD-sized workspace is large enough for every entry point.
 * The first 256 bytes hold the device error word; zero the whole workspace
 * once after allocating it (moe_get_device_error() re-zeroes the word). */
size_t moe_workspace_bytes(const moe_dims_t* d, moe_ws_kind_t which);

/* Router logits z = x W_r^T + o (the score whose sigmoid is the affinity,
 * "02 · DeepSeek-V3" §1.3 eq. 15), fp32 accumulation of exact products.
 * x [T, H] bf16, w_router [E, H] fp32, router_offset [E] fp32 or NULL
 * (o = 0) -> logits [T, E] fp32; the offset is added once, in fp32, after
 * the accumulation.  When E % 16 == 0 it runs on the tensor cores: W_r is
 * split exactly into three bf16 parts (hi + mid + lo == W_r) in the
 * workspace and the three products are accumulated into one fp32
 * accumulator; with few 128-token tiles (a decode batch) the sum over H is
 * split into ranges whose fp32 partial sums, kept in the workspace, are
 * added in range order (deterministic).  Otherwise an fp32 SIMT kernel.
 * Workspace: MOE_WS_ROUTER_LOGITS. */
moe_status_t moe_router_logits(const moe_dims_t* d, const uint16_t* x,
                               const float* w_router,
                               const float* router_offset, float* logits,
                               void* ws, size_t ws_bytes,
                               moe_stream_t stream);

/* The router weight's exact three-way bf16 split, done once for weights
 * that do not change between calls: w_router [E, H] fp32 -> split
 * [3, E, H] bf16 (hi, mid, lo; hi + mid + lo == w_router for every normal
 * value, the parts moe_router_logits forms in its workspace).  E % 16 == 0
 * (the tensor-core path; MOE_ERR_UNSUPPORTED otherwise), H > 0.  Pass the
 * result as moe_weights_t.router_split.  Needs no workspace. */
moe_status_t moe_router_weight_split(const float* w_router, int32_t E,
                                     int32_t H, uint16_t* split,
                                     moe_stream_t stream);

/* Routing from precomputed logits ("02 · DeepSeek-V3" §1.3, §1.4):
 * sigmoid, + bias for selection, group-limited top-K, gates renormalised
 * over the chosen K, and the per-expert load histogram.
 *   logits   [T, E] fp32      in
 *   bias     [E]    fp32      in (not modified)
 *   topk_idx [T, K] int32     out, slot k = k-th largest s+b among the kept
 *                             groups' experts (ties: lower expert index)
 *   topk_gate[T, K] fp32      out, s_{e_k} / sum_j s_{e_j}, summed in slot
 *                             order (sum to 1)
 *   counts   [E]    int32     out, tokens routed to each expert
 * The fp32 sigmoid is one fixed sequence of correctly rounded operations
 * (Cody-Waite reduction, degree-7 Taylor polynomial, correctly rounded
 * reciprocal of 1 + e), so routing is reproducible bit for bit.
 * Workspace: MOE_WS_ROUTE. */
moe_status_t moe_route(const moe_dims_t* d, const float* logits,
                       const float* bias, int32_t* topk_idx, float* topk_gate,
                       int32_t* counts, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* moe_route without a workspace argument, for callers that cannot give
 * this library any device memory beyond inputs and outputs -- for example a
 * plugin whose host framework owns all device allocations and offers no
 * scratch, or a loop that must not call cudaMalloc after start-up because
 * it synchronises the device.  (The pages have no counterpart: this is an
 * interface variant, not part of the method.)  Results are identical to
 * moe_route's.  Its scratch is one static device array of 1.6 MiB (412672
 * int32) that every GPU loading this library holds until the process
 * exits; it allocates nothing and calls no allocating routine.
 *   Limit: ceil(T/64) * E <= 262144 (T <= 65536 at E = 256), else
 *   MOE_ERR_WORKSPACE before anything is launched.
 *   The first call in a CUDA context looks up the array's device address
 *   (one cudaGetSymbolAddress per context, so a context re-created after
 *   cudaDeviceReset gets its own lookup); make that first call before any
 *   stream capture.
 *   All calls share the array: calls whose kernels overlap on the GPU (on
 *   different streams, or from several threads) race on it and must be
 *   serialised by the caller.  Nothing in it needs clearing between calls. */
moe_status_t moe_route_static_scratch(const moe_dims_t* d, const float* logits,
                                      const float* bias, int32_t* topk_idx,
                                      float* topk_gate, int32_t* counts,
                                      moe_stream_t stream);

/* Dispatch order and token gather (the single-GPU form of the pages'
 * "dispatch" step, "02 · DeepSeek-V3" §2 and §5.1).  A stable counting sort
 * of the (token, slot) pairs by expert:
 *   offsets [E+1]  int32  out, offsets[e] = sum_{e'<e} c_e', offsets[E]=T*K
 *   dest    [T, K] int32  out, row of (t, k) in the expert-sorted order:
 *                         offsets[e] + #{t' < t that chose e}
 *   src_row [T*K]  int32  out, inverse of dest: src_row[dest[t,k]] = t*K+k
 *   xp      [T*K, H] bf16 out, xp[dest[t,k]] = x[t]; may be NULL (indices
 *                         only), x may then be NULL too.
 * topk_idx must hold valid, per-token distinct experts (as moe_route
 * writes them).  Workspace: MOE_WS_PERMUTE. */
moe_status_t moe_permute(const moe_dims_t* d, const uint16_t* x,
                         const int32_t* topk_idx, int32_t* offsets,
                         int32_t* dest, int32_t* src_row, uint16_t* xp,
                         void* ws, size_t ws_bytes, moe_stream_t stream);

/* Expert FFNs ("02 · DeepSeek-V3" §1.1: SwiGLU, three matrices per expert)
 * as grouped BF16 GEMMs on the tcgen05 tensor cores, fp32 accumulation in
 * tensor memory, SwiGLU fused into the first GEMM's epilogue; the
 * intermediate is stored as bf16.
 *   xp      [T*K, H] bf16  routed rows, expert e owns rows
 *                          [offsets[e], offsets[e+1])
 *   x       [T, H]   bf16  token rows for the shared expert
 *   offsets [E+1]    int32 as written by moe_permute (read on the device)
 *   yp      [T*K, H] bf16  out, FFN_e(row) for every routed row (ungated)
 *   ys      [T, H]   bf16  out, FFN_shared(x_t)
 * Workspace: MOE_WS_EXPERT_FFN.  The intermediate h = silu(p) * q of the
 * routed rows, [T*K, I] bf16, is left in a MOE_WS_EXPERT_FFN workspace at
 * byte offset 256 until the next call (for inspection). */
moe_status_t moe_expert_ffn(const moe_dims_t* d, const moe_weights_t* w,
                            const uint16_t* xp, const uint16_t* x,
                            const int32_t* offsets, uint16_t* yp,
                            uint16_t* ys, void* ws, size_t ws_bytes,
                            moe_stream_t stream);

/* Routed experts only: the grouped SwiGLU FFNs of moe_expert_ffn over
 * R = d->T * d->topk expert-sorted rows, without the shared expert -- the
 * receive side of expert parallelism ("02 · DeepSeek-V3" §5.1: a device
 * runs its own experts on the rows other devices sent it); pass d->T = R,
 * d->topk = 1 for R received rows and d->E = the device's experts.
 *   xp [R, H] bf16, offsets [E+1] int32 (device; offsets[E] <= R),
 *   yp [R, H] bf16 out.  Only w->w1, w3, w2 are read (others may be NULL).
 * Nothing is routed here, so the routing shape rules do not apply: any
 * E >= 1 (<= 1024); n_group and topk_group are not read.  (The shared
 * expert can run through this call too, as one expert over the tokens.)
 * Workspace: MOE_WS_EXPERT_FFN (its shared-expert part is unused), which
 * moe_workspace_bytes sizes for such dims as well. */
moe_status_t moe_expert_ffn_routed(const moe_dims_t* d, const moe_weights_t* w,
                                   const uint16_t* xp, const int32_t* offsets,
                                   uint16_t* yp, void* ws, size_t ws_bytes,
                                   moe_stream_t stream);

/* Expert parallelism: the receive-side row order ("02 · DeepSeek-V3" §1.3
 * node-limited routing, §2 and §5.1 dispatch / combine across devices).
 * Device r holds experts [r*El, (r+1)*El); the rows it receives arrive
 * from each source device s in order, each source's rows sorted by expert
 * ("source-major").  moe_ep_plan maps them to "expert-major" order (expert
 * l's rows from source 0, 1, ... together, the grouped GEMM's segments):
 *   counts [n_src, n_local] int32 (device): rows source s sends for local
 *          expert l (the sources' moe_route counts of these experts)
 *   rows   = sum of counts (the host knows it: it sized the exchange)
 *   perm   [rows] int32 out: expert-major row of source-major row i
 *   offsets_local [n_local + 1] int32 out: expert-major segment starts
 * n_src * n_local <= 4096 (MOE_ERR_UNSUPPORTED beyond).  A sum of counts
 * other than rows records MOE_ERR_DEVICE_BOUNDS in the error word of ws
 * (any workspace; may be NULL: nothing recorded).
 * moe_ep_permute_rows moves rows of row_bytes (any width) by such
 * a map: inverse = 0: out[perm[i]] = in[i] (source-major -> expert-major);
 * inverse = 1: out[i] = in[perm[i]] (back, for the return trip).  in and
 * out may not alias. */
moe_status_t moe_ep_plan(int32_t n_src, int32_t n_local, const int32_t* counts,
                         int64_t rows, int32_t* perm, int32_t* offsets_local,
                         void* ws, moe_stream_t stream);
moe_status_t moe_ep_permute_rows(const void* in, int64_t rows,
                                 int64_t row_bytes, const int32_t* perm,
                                 int32_t inverse, void* out, void* ws,
                                 moe_stream_t stream);

/* Combine (eq. 12): out_t = bf16( x_t + ys_t + sum_k g_{t,k} yp[dest[t,k]] ),
 * fp32 arithmetic, slots summed in order.  out [T, H] bf16 may not alias
 * the inputs.  A slot whose dest lies outside [0, T*K) (moe_permute writes
 * -1 for an invalid expert id) contributes nothing: its yp row is not read.
 * Needs no workspace. */
moe_status_t moe_combine(const moe_dims_t* d, const uint16_t* x,
                         const uint16_t* ys, const uint16_t* yp,
                         const int32_t* dest, const float* topk_gate,
                         uint16_t* out, moe_stream_t stream);

/* Auxiliary-loss-free bias step ("02 · DeepSeek-V3" §1.4), in place:
 * b_e -= gamma if c_e*E > T*K (overloaded), b_e += gamma if c_e*E < T*K,
 * unchanged at exactly the mean load.  counts [E] int32 in, bias [E] fp32
 * in/out, load_stats [3] fp32 out (max, mean, min of c) or NULL.
 * Call it after the step's routing: the next step routes with the new b. */
moe_status_t moe_bias_update(const moe_dims_t* d, const int32_t* counts,
                             float* bias, float* load_stats,
                             moe_stream_t stream);

/* Sequence-wise balance loss, forward value ("02 · DeepSeek-V3" §1.4,
 * eq. 17-20: the small complementary loss kept beside the bias, alpha =
 * 1e-4 for V3).  The T tokens are cut into sequences of seq_len
 * consecutive tokens (the last one holds the remainder), n_seq =
 * ceil(T / seq_len).  For a sequence of T_s tokens:
 *   s'_{t,i} = s_{t,i} / sum_j s_{t,j}    (s = the routing sigmoid of z)
 *   P_i = (1/T_s) sum_t s'_{t,i}
 *   c_i = #{t : i is among the topk largest s_{t,.}} -- the raw affinity
 *         over all E experts: no bias, no group limit (ties: lower index)
 *   f_i = E c_i / (topk T_s),   L = alpha sum_i f_i P_i
 *   logits     [T, E]      fp32 in
 *   counts_seq [n_seq, E]  int32 out, c_i per sequence (exact)
 *   P_seq      [n_seq, E]  fp32  out
 *   loss       [n_seq]     fp32  out
 * fp32 arithmetic in a fixed order (per token: lane partial sums, then a
 * butterfly; per sequence: up to ceil(seq_len/256) row splits, each cut
 * into 32 token ranges summed in token order, the ranges and then the
 * splits added in order), so results are reproducible run to run.
 * seq_len < 1 or a non-finite alpha: MOE_ERR_INVALID_ARG.  n_group and
 * topk_group are validated but not used.  Workspace: MOE_WS_SEQ_BALANCE. */
moe_status_t moe_seq_balance_loss(const moe_dims_t* d, const float* logits,
                                  int32_t seq_len, float alpha,
                                  int32_t* counts_seq, float* P_seq,
                                  float* loss, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* Backward of routing to the router logits (the training side of
 * "02 · DeepSeek-V3" §1.4).  The top-K choices and the balance loss's
 * indicator counts are piecewise constant in z and carry no gradient; the
 * bias is not part of backpropagation (the page says so).  s is the
 * forward's sigmoid.  Both write dlogits [T, E] fp32, or add to it when
 * accumulate != 0 (so the two can be summed in place).
 *
 * moe_route_backward: the gates g_k = s_k / D (D = sum of the chosen s):
 *   dlogits[t, m] = s_m (1 - s_m) / D * (dgate[t, m] - sum_k dgate_k g_k)
 * for each chosen expert m = topk_idx[t, k], 0 for the others.
 *   logits [T, E], topk_idx [T, K] (as moe_route wrote it), dgate [T, K]
 *   the upstream gradient of the gates.  An expert id outside [0, E) is
 *   skipped and records MOE_ERR_DEVICE_BOUNDS in the workspace error word.
 *   Workspace: MOE_WS_ROUTE (only its error word is used). */
moe_status_t moe_route_backward(const moe_dims_t* d, const float* logits,
                                const int32_t* topk_idx, const float* dgate,
                                int accumulate, float* dlogits, void* ws,
                                size_t ws_bytes, moe_stream_t stream);

/* moe_seq_balance_loss_backward: the sequence-wise balance loss (eq. 17-20)
 * with the forward's counts (moe_seq_balance_loss's counts_seq [n_seq, E])
 * and an upstream gradient dloss [n_seq] per sequence (NULL = 1):
 *   dlogits[t, i] = dloss_q alpha / T_s * s_i (1 - s_i) / S_t
 *                   * (f_i - sum_j f_j s_j / S_t),
 *   S_t = sum_j s_t,j, f_i = E c_i / (topk T_s).
 * Needs no workspace. */
moe_status_t moe_seq_balance_loss_backward(const moe_dims_t* d,
                                           const float* logits,
                                           int32_t seq_len, float alpha,
                                           const int32_t* counts_seq,
                                           const float* dloss, int accumulate,
                                           float* dlogits,
                                           moe_stream_t stream);

/* moe_route_balance_backward: both of the above in one pass, for a
 * training step that backpropagates the gates and the sequence-wise
 * balance loss through the same logits: dlogits = (dlogits when
 * accumulate != 0, else 0) + the gates' term of moe_route_backward + the
 * balance term of moe_seq_balance_loss_backward, added in that order, so
 * the result equals moe_route_backward followed by
 * moe_seq_balance_loss_backward with accumulate set, bit for bit.  Each
 * logits row is read once and each sigmoid taken once.  Arguments as in
 * those two calls; an expert id outside [0, E) is skipped and records
 * MOE_ERR_DEVICE_BOUNDS in the workspace error word.
 * Workspace: MOE_WS_ROUTE (only its error word is used). */
moe_status_t moe_route_balance_backward(const moe_dims_t* d,
                                        const float* logits,
                                        const int32_t* topk_idx,
                                        const float* dgate, int32_t seq_len,
                                        float alpha,
                                        const int32_t* counts_seq,
                                        const float* dloss, int accumulate,
                                        float* dlogits, void* ws,
                                        size_t ws_bytes, moe_stream_t stream);

/* FP8 (E4M3) fine-grained quantization ("02 · DeepSeek-V3" §2, mixed
 * precision): every group of 128 x 128 weights or 1 x 128 activations
 * (one row, 128 channels) gets its own fp32 scale from the group's max
 * |value|, taken online:
 *   s = amax / 448 (correctly rounded; s = 1 for an all-zero group)
 *   code = the E4M3 value nearest to the fp32 quotient x / s, ties to
 *          the even mantissa, saturated to +-448 (448 = largest E4M3)
 * Codes are E4M3 bytes (sign, 4-bit exponent with bias 7, 3-bit
 * mantissa); value = E4M3(code) * s.  Rows and columns are bf16 inputs,
 * row-major; rows = 0 is valid and does nothing.
 *
 * moe_quantize_fp8_blocks: w [rows, cols] bf16 -> q [rows, cols] u8 and
 *   scale [rows/128, cols/128] fp32 (block (i, j) at scale[i*cols/128+j]).
 *   rows, cols multiples of 128 (MOE_ERR_INVALID_ARG otherwise); rows/128
 *   <= 65535.  For the experts' weights pass [E*I, H] (w1, w3) and
 *   [E*H, I] (w2): with I and H multiples of 128 no block straddles two
 *   experts.  Needs no workspace. */
moe_status_t moe_quantize_fp8_blocks(const uint16_t* w, int64_t rows,
                                     int64_t cols, uint8_t* q, float* scale,
                                     moe_stream_t stream);

/* moe_quantize_fp8_rows: x [rows, cols] bf16 -> q [rows, cols] u8 and
 * scale [rows, cols/128] fp32, one scale per 1 x 128 tile.  cols a multiple
 * of 128.  Needs no workspace. */
moe_status_t moe_quantize_fp8_rows(const uint16_t* x, int64_t rows,
                                   int64_t cols, uint8_t* q, float* scale,
                                   moe_stream_t stream);

/* Quantise-on-permute: the tokens are quantized before dispatch, and the
 * dispatch moves FP8 rows ("02 · DeepSeek-V3" §2: activations are cast to
 * FP8 before they are sent).  x [T, H] bf16 (H % 128 == 0, else
 * MOE_ERR_UNSUPPORTED) is quantized in 1 x 128 tiles once:
 *   xq [T, H] u8, xs [T, H/128] fp32            the token rows (shared expert)
 *   xpq[dest[t,k]] = xq[t], xps[dest[t,k]] = xs[t]  the expert-sorted rows
 *                  ([T*K, H] u8 and [T*K, H/128] fp32)
 * dest [T, K] as written by moe_permute (which may be called with xp =
 * NULL for the indices alone).  A dest row outside [0, T*K) is skipped and
 * records MOE_ERR_DEVICE_BOUNDS in the workspace error word.
 * Workspace: MOE_WS_PERMUTE (only its error word is used). */
moe_status_t moe_permute_fp8(const moe_dims_t* d, const uint16_t* x,
                             const int32_t* dest, uint8_t* xq, float* xs,
                             uint8_t* xpq, float* xps, void* ws,
                             size_t ws_bytes, moe_stream_t stream);

/* FP8 expert weights: E4M3 codes and 128 x 128 block scales as
 * moe_quantize_fp8_blocks writes them (device pointers, caller-owned):
 *   w1, w3 [E*I, H] codes, w1_scale, w3_scale [E*I/128, H/128]
 *   w2     [E*H, I] codes, w2_scale          [E*H/128, I/128]
 *   ws1, ws3 [I_s, H], ws1_scale, ws3_scale [I_s/128, H/128] (shared)
 *   ws2    [H, I_s],   ws2_scale            [H/128, I_s/128] */
typedef struct {
  const uint8_t* w1;
  const float* w1_scale;
  const uint8_t* w3;
  const float* w3_scale;
  const uint8_t* w2;
  const float* w2_scale;
  const uint8_t* ws1;
  const float* ws1_scale;
  const uint8_t* ws3;
  const float* ws3_scale;
  const uint8_t* ws2;
  const float* ws2_scale;
} moe_weights_fp8_t;

/* Expert FFNs in FP8 ("02 · DeepSeek-V3" §2 mixed precision on §1.1's
 * SwiGLU experts): E4M3 x E4M3 products on the tcgen05 tensor cores, each
 * 128-element slice of the reduction (one scale group of both operands)
 * summed on its own in fp32 and promoted into fp32 registers times its
 * activation and weight scales; the intermediate silu(p) * q is quantized
 * to E4M3 in 1 x 128 tiles for the down projection.
 *   xpq [T*K, H] u8, xps [T*K, H/128] fp32   routed rows (moe_permute_fp8)
 *   xq  [T, H] u8,   xs  [T, H/128] fp32     token rows (shared expert)
 *   offsets [E+1] int32                      as written by moe_permute
 *   yp [T*K, H] bf16 out, FFN_e(row) for every routed row (ungated)
 *   ys [T, H] bf16 out, FFN_shared(x_t)
 * H, I, I_shared must be multiples of 128 and at most 8192
 * (MOE_ERR_UNSUPPORTED otherwise).  Its tiles hold up to 32 token rows:
 * it is built for batches where each expert sees few tokens (decode), whose
 * time is the weight stream that FP8 halves.
 * Workspace: MOE_WS_EXPERT_FFN_FP8. */
moe_status_t moe_expert_ffn_fp8(const moe_dims_t* d, const moe_weights_fp8_t* w,
                                const uint8_t* xpq, const float* xps,
                                const uint8_t* xq, const float* xs,
                                const int32_t* offsets, uint16_t* yp,
                                uint16_t* ys, void* ws, size_t ws_bytes,
                                moe_stream_t stream);

/* FP8 with power-of-two group scales ("02 · DeepSeek-V3" §2 likens its
 * 1 x 128 / 128 x 128 groups to the microscaling formats whose scaling
 * Blackwell's tensor cores apply natively; there a scale is a power of two
 * held as an 8-bit exponent).  Same groups and codes as the FP8 calls
 * above, but each group's scale is
 *   s = 2^e, e the least integer with 448 * 2^e >= amax (amax = the
 *       group's max |value|), at least -127; e = 0 for an all-zero group
 * stored as the byte e + 127 (UE8M0), and
 *   code = the E4M3 value nearest to x / s (exact quotient), ties to the
 *          even mantissa, saturated to +-448.
 * moe_quantize_mx_blocks: w [rows, cols] bf16 -> q [rows, cols] u8 and
 *   scale [rows/128, cols/128] u8; sizes and errors as
 *   moe_quantize_fp8_blocks.
 * moe_quantize_mx_rows: x [rows, cols] bf16 -> q u8 and scale
 *   [rows, cols/128] u8, one per 1 x 128 tile; as moe_quantize_fp8_rows.
 * moe_permute_mx: quantise-on-permute as moe_permute_fp8 with these
 *   scales: xq [T, H] u8, xs [T, H/128] u8, xpq[dest[t,k]] = xq[t],
 *   xps[dest[t,k]] = xs[t]; workspace MOE_WS_PERMUTE (error word only). */
moe_status_t moe_quantize_mx_blocks(const uint16_t* w, int64_t rows,
                                    int64_t cols, uint8_t* q, uint8_t* scale,
                                    moe_stream_t stream);
moe_status_t moe_quantize_mx_rows(const uint16_t* x, int64_t rows,
                                  int64_t cols, uint8_t* q, uint8_t* scale,
                                  moe_stream_t stream);
moe_status_t moe_permute_mx(const moe_dims_t* d, const uint16_t* x,
                            const int32_t* dest, uint8_t* xq, uint8_t* xs,
                            uint8_t* xpq, uint8_t* xps, void* ws,
                            size_t ws_bytes, moe_stream_t stream);

/* Expert weights with power-of-two scales: E4M3 codes and UE8M0 block
 * scales as moe_quantize_mx_blocks writes them (device pointers,
 * caller-owned), shapes as moe_weights_fp8_t. */
typedef struct {
  const uint8_t* w1;
  const uint8_t* w1_scale;
  const uint8_t* w3;
  const uint8_t* w3_scale;
  const uint8_t* w2;
  const uint8_t* w2_scale;
  const uint8_t* ws1;
  const uint8_t* ws1_scale;
  const uint8_t* ws3;
  const uint8_t* ws3_scale;
  const uint8_t* ws2;
  const uint8_t* ws2_scale;
} moe_weights_mx_t;

/* Expert FFNs in FP8 with power-of-two group scales, scaled by the tensor
 * cores ("02 · DeepSeek-V3" §2 mixed precision on §1.1's SwiGLU experts):
 * tcgen05 block-scaled MMAs multiply every 32-element slice of a product by
 * its token's and its weight block's scale and accumulate the whole
 * reduction in fp32, so no partial sum is promoted on the CUDA cores; the
 * intermediate silu(p) * q is quantized to E4M3 in 1 x 128 tiles with
 * power-of-two scales for the down projection.
 *   xpq [T*K, H] u8, xps [T*K, H/128] u8    routed rows (moe_permute_mx)
 *   xq  [T, H] u8,   xs  [T, H/128] u8      token rows (shared expert)
 *   offsets [E+1] int32                     as written by moe_permute
 *   yp [T*K, H] bf16 out, FFN_e(row) for every routed row (ungated)
 *   ys [T, H] bf16 out, FFN_shared(x_t)
 * H, I, I_shared must be multiples of 128 (MOE_ERR_UNSUPPORTED otherwise).
 * Token chunks of up to 192 rows (224 when the experts average 256 rows or
 * more), so one weight tile serves a prefill expert's rows at once.
 * Workspace: MOE_WS_EXPERT_FFN_MX. */
moe_status_t moe_expert_ffn_mx(const moe_dims_t* d, const moe_weights_mx_t* w,
                               const uint8_t* xpq, const uint8_t* xps,
                               const uint8_t* xq, const uint8_t* xs,
                               const int32_t* offsets, uint16_t* yp,
                               uint16_t* ys, void* ws, size_t ws_bytes,
                               moe_stream_t stream);

/* The routed experts alone in FP8 with power-of-two scales, over any
 * number of expert-sorted rows: expert parallelism's receive side when the
 * rows are dispatched as E4M3 codes ("02 · DeepSeek-V3" §2: activations
 * are cast to FP8 before dispatch, the expert outputs return in BF16).
 * d->T = the rows R, d->topk = 1, d->E = the local experts; d's routing
 * fields are not used.  xpq [R, H] u8, xps [R, H/128] u8 (UE8M0), offsets
 * [E+1], yp [R, H] bf16 out.  w->w1, w3, w2 and their scales as in
 * moe_expert_ffn_mx (the shared pointers are not read; the shared expert
 * can run through this call as one expert over the tokens).
 * Workspace: MOE_WS_EXPERT_FFN_MX, which moe_workspace_bytes sizes for
 * such dims as well. */
moe_status_t moe_expert_ffn_mx_routed(const moe_dims_t* d,
                                      const moe_weights_mx_t* w,
                                      const uint8_t* xpq, const uint8_t* xps,
                                      const int32_t* offsets, uint16_t* yp,
                                      void* ws, size_t ws_bytes,
                                      moe_stream_t stream);

/* Backward of the expert FFNs and the combine, for a fixed routing (the
 * training side of "02 · DeepSeek-V3" §1.1 SwiGLU experts and §1.3 eq. 12;
 * §1.4 trains the layer, §2 keeps the master weights and their gradients
 * in higher precision than the GEMM inputs).  For the layer output
 *   out_t = x_t + FFN_s(x_t) + sum_k g_{t,k} FFN_{e_k}(x_t)
 * and its upstream gradient dout [T, H] (bf16):
 *   dgate [T, K] fp32  dgate[t,k] = <dout_t, FFN_{e_k}(x_t)>, the input of
 *                      moe_route_backward
 *   dx    [T, H] bf16  dout_t + (shared expert's input gradient of dout_t)
 *                      + sum_k (expert e_k's input gradient of g dout_t);
 *                      the path through the router logits is not included
 *                      (moe_route_backward gives dlogits; dlogits W_r is the
 *                      caller's)
 *   dw1, dw3 [E, I, H], dw2 [E, H, I], dws1, dws3 [I_s, H], dws2 [H, I_s]
 *                      fp32: the weight gradients; written, or added to the
 *                      arrays' contents when accumulate != 0 (gradient
 *                      accumulation over micro-batches).  An expert that no
 *                      token chose gets a zero gradient (or is left as it
 *                      is when accumulating).
 * x [T, H] bf16, topk_idx / topk_gate [T, K] as moe_route wrote them (valid,
 * per-token distinct experts), weights as for moe_forward (w_router and
 * router_offset are not used).  p = W1 a, q = W3 a and silu(p) q are
 * recomputed on the tensor cores with fp32 accumulation; the intermediate
 * gradients dp, dq and the rows g dout are bf16 GEMM operands, every GEMM
 * accumulates in fp32.  H, I, I_shared multiples of 64; H <= 16384.
 * Workspace: MOE_WS_EXPERT_BWD (it holds the recomputed p, q in fp32 and
 * the rows dispatched to 16-row-aligned expert segments). */
moe_status_t moe_expert_backward(const moe_dims_t* d, const moe_weights_t* w,
                                 const uint16_t* x, const uint16_t* dout,
                                 const int32_t* topk_idx,
                                 const float* topk_gate, int accumulate,
                                 uint16_t* dx, float* dgate, float* dw1,
                                 float* dw3, float* dw2, float* dws1,
                                 float* dws3, float* dws2, void* ws,
                                 size_t ws_bytes, moe_stream_t stream);

/* Redundant-expert placement ("02 · DeepSeek-V3" §5.1: high-load experts
 * are replicated from online load statistics, e.g. 32 redundant experts
 * with one extra expert per GPU, revised periodically).  HOST function:
 * all pointers are host memory, nothing is launched; it plans between
 * steps from a count vector the caller read back (e.g. moe_forward's
 * counts_out summed over the statistics window).
 *   load [E] int64            tokens routed to each expert (>= 0)
 *   n_devices D, slots_per_device r; E % D == 0
 *   slot_expert [D * r] int32 out: the expert copied into slot (d, s) at
 *                             [d*r + s], -1 = left empty
 *   device_load [D] int64     out: each device's load after planning
 * Base placement: device d hosts experts [d*E/D, (d+1)*E/D).  An expert
 * with a copy serves its c tokens round-robin: the original keeps
 * ceil(c/2), the copy floor(c/2).  Experts are taken heaviest first (load
 * desc, index asc) while slots are free and loads positive; each copy goes
 * to the least-loaded device (ties: lower index) with a free slot other
 * than the expert's own; an expert whose only free slots are on its own
 * device is passed over.  MOE_ERR_INVALID_ARG on a NULL pointer (slot_expert
 * may be NULL when D * r == 0), E % D != 0, or a negative load. */
moe_status_t moe_plan_redundant_experts(const int64_t* load, int32_t E,
                                        int32_t n_devices,
                                        int32_t slots_per_device,
                                        int32_t* slot_expert,
                                        int64_t* device_load);

/* The whole layer forward in one call: router logits, routing, dispatch,
 * expert FFNs, combine, and -- if update_bias != 0 -- the bias step on this
 * batch's load (applied after routing, so this call routes with the bias it
 * was given).  It allocates nothing and never synchronises, so a step can be
 * captured into a CUDA graph and replayed (the tests capture it after one
 * ordinary call on the device, and check the replay bit for bit).
 *   x [T, H] bf16 in; bias [E] fp32 in (in/out when update_bias);
 *   out [T, H] bf16 out.
 *   Optional outputs (NULL = not written): logits_out [T, E] fp32,
 *   topk_idx_out [T, K] int32, topk_gate_out [T, K] fp32, counts_out [E]
 *   int32, load_stats_out [3] fp32.
 * Workspace: MOE_WS_FORWARD. */
moe_status_t moe_forward(const moe_dims_t* d, const moe_weights_t* w,
                         const uint16_t* x, float* bias, int update_bias,
                         uint16_t* out, float* logits_out,
                         int32_t* topk_idx_out, float* topk_gate_out,
                         int32_t* counts_out, float* load_stats_out, void* ws,
                         size_t ws_bytes, moe_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status_t s);

/* Synchronises `stream`, reads and clears the device error word at the
 * start of `ws`, and returns it (MOE_OK if no kernel recorded an error).
 * Meant for tests and debugging: it blocks the host. */
moe_status_t moe_get_device_error(void* ws, moe_stream_t stream);

/* Upper bound, in nanoseconds, on every device-side wait of the GEMM
 * kernels (default 2e9 ns).  0 restores the default.  Takes effect for
 * launches made after the call; not thread-safe against concurrent
 * launches. */
void moe_set_wait_timeout_ns(uint64_t ns);

/* Number of persistent CTAs of the expert GEMM kernels: n > 0 caps the
 * grid at n CTAs (at most one per SM), 0 restores one CTA per SM (the
 * default).  Results do not depend on it -- every CTA walks the same unit
 * list with a stride of the grid size -- so it serves tuning and tests that
 * must drive many units, and both kinds of tensor-memory slot use, through
 * one CTA.  Takes effect for launches made after the call; not thread-safe
 * against concurrent launches. */
void moe_set_gemm_ctas(int32_t n);

/* Profiling hook for kernel-level timing.  When `events` is non-NULL and
 * n >= MOE_FORWARD_KERNELS + 1, moe_forward records events[i] (cudaEvent_t
 * handles created by the caller, passed as void*) on its stream just before
 * its i-th kernel launch, and events[MOE_FORWARD_KERNELS] after the last,
 * so consecutive events bracket one kernel each.  The launch order is:
 *   0 router logits (weight split + GEMM), 1 route, 2 count scan (+bias
 *   step), 3 dispatch order,
 *   4 gather, 5 expert up-projection GEMM (+SwiGLU), 6 expert
 *   down-projection GEMM, 7 combine.
 * NULL / n = 0 disables.  The array must stay valid while enabled.  Global
 * state: not for concurrent use from several threads. */
#define MOE_FORWARD_KERNELS 8
/* While enabled, moe_expert_backward records events[0..6] of the same array
 * around its six stages: 0 padded dispatch (3 kernels), 1 recompute of p,
 * q (GEMM), 2 dgrad of the down projection (GEMM), 3 dgrad of the up
 * projections (GEMM), 4 weight gradients (GEMM), 5 token and gate
 * gradients, and events[6] after the last. */
#define MOE_BACKWARD_STAGES 6
void moe_set_profile_events(void* const* events, int32_t n);

/* MOE_ABI_VERSION of the loaded library. */
int32_t moe_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DEEPSEEKMOE_B300_MOE_H */
