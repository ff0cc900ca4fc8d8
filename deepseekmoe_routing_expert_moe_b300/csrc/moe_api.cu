// C ABI of libmoe: host-side validation, workspace layout and the launch
// sequences of the DeepSeekMoE layer forward (include/moe.h documents
// every entry point).  Nothing here allocates device memory or
// synchronises, except moe_get_device_error().
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/moe.h"
#include "device_common.cuh"
#include "internal.h"

namespace {

using moe::DevStatus;

constexpr size_t kAlign = 256;
constexpr size_t kStatusBytes = 256;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
uint64_t g_wait_limit_ns = kDefaultWaitNs;
void* const* g_prof_events = nullptr;  // moe_set_profile_events()

// records profiling event i (if enabled) on stream s
inline void prof_mark(int i, cudaStream_t s) {
  if (g_prof_events != nullptr)
    cudaEventRecord(static_cast<cudaEvent_t>(g_prof_events[i]), s);
}

inline size_t up(size_t b) { return (b + kAlign - 1) / kAlign * kAlign; }
inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}
inline cudaStream_t cs(moe_stream_t s) { return static_cast<cudaStream_t>(s); }

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

// Shape checks of the expert GEMMs alone (no routing: any E >= 1).
moe_status_t check_ffn_only_dims(const moe_dims_t* d) {
  if (d == nullptr) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->H <= 0 || d->E <= 0 || d->topk <= 0 || d->I <= 0 ||
      d->I_shared <= 0)
    return MOE_ERR_INVALID_ARG;
  if ((long long)d->T * (d->topk + 1) >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  if (d->H % 64 != 0 || d->I % 64 != 0 || d->I_shared % 64 != 0)
    return MOE_ERR_UNSUPPORTED;
  if (d->E > 1024 || (long long)d->E * d->I >= (1ll << 31) ||
      (long long)d->E * d->H >= (1ll << 31))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// Shape checks shared by every entry point.
moe_status_t check_dims(const moe_dims_t* d, bool need_ffn) {
  if (d == nullptr) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->H <= 0 || d->E <= 0 || d->n_group <= 0 ||
      d->topk_group <= 0 || d->topk <= 0)
    return MOE_ERR_INVALID_ARG;
  if (d->E % d->n_group != 0) return MOE_ERR_INVALID_ARG;
  const int gs = d->E / d->n_group;
  if (gs < 2) return MOE_ERR_INVALID_ARG;  // the group score needs a top-2
  if (d->topk_group > d->n_group) return MOE_ERR_INVALID_ARG;
  if (d->topk > d->topk_group * gs) return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(d->gamma)) return MOE_ERR_INVALID_ARG;
  if ((long long)d->T * (d->topk + 1) >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  // routing kernel shape rules
  if (d->E > 1024 || (d->E > 32 && d->E % 32 != 0)) return MOE_ERR_UNSUPPORTED;
  if (d->n_group > 32 || d->topk > 32) return MOE_ERR_UNSUPPORTED;
  const int epl = d->E <= 32 ? 1 : d->E / 32;  // experts per lane
  if (!is_pow2(epl) || gs % epl != 0 || !is_pow2(gs / epl))
    return MOE_ERR_UNSUPPORTED;
  if (d->H % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (d->H / 8 > 128 * 16) return MOE_ERR_UNSUPPORTED;  // gather row limit
  if (need_ffn) {
    if (d->I <= 0 || d->I_shared <= 0) return MOE_ERR_INVALID_ARG;
    if (d->I % 64 != 0 || d->I_shared % 64 != 0) return MOE_ERR_UNSUPPORTED;
    if ((long long)d->E * d->I >= (1ll << 31) ||
        (long long)d->E * d->H >= (1ll << 31))
      return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

// ----------------------------------------------------------- workspace
struct Layout {
  size_t status = 0;  // always at 0
  size_t block_counts = 0, block_base = 0;
  size_t logits = 0, idx = 0, gate = 0, counts = 0, offsets = 0, dest = 0,
         src_row = 0;
  size_t xp = 0, h = 0, hs = 0, yp = 0, ys = 0;
  size_t w_split = 0;  // [3, E, H] bf16 parts of the router weight
  size_t r_partial = 0;  // [ksplit, T, E] fp32 partial router sums
  size_t bal_sp = 0, bal_flags = 0;  // [T, E] fp32 s', [T, E] u8 top-K flags
  size_t bal_pP = 0, bal_pc = 0;     // per-split partial sums (bounded)
  size_t f8_mq = 0, f8_ms = 0, f8_msq = 0, f8_mss = 0;  // FP8 intermediate
  size_t mx_mq = 0, mx_ms = 0, mx_msq = 0, mx_mss = 0;  // its UE8M0 form
  // expert backward (padded dispatch of cap rows)
  size_t b_poff = 0, b_ticket = 0, b_pdest = 0, b_gp = 0, b_xpp = 0, b_dpp = 0, b_p = 0,
         b_q = 0, b_hg = 0, b_dp = 0, b_dq = 0, b_dgp = 0, b_dxpp = 0,
         b_ps = 0, b_qs = 0, b_hgs = 0, b_dps = 0, b_dqs = 0, b_dxs = 0;
  size_t total = 0;
};

// moe_forward gathers the routed rows from x inside the up GEMM (TMA
// gather4, four 128-byte rows per copy) when the experts see few rows each;
// with more rows per expert the gathers' issue rate would bound the GEMM,
// and the rows are copied out once (expert-sorted) instead.
constexpr long long kGatherMeanRows = 64;
bool gather_rows(const moe_dims_t* d) {
  return (long long)d->T * d->topk < kGatherMeanRows * d->E;
}

Layout layout(const moe_dims_t* d, moe_ws_kind_t which) {
  Layout L;
  size_t o = kStatusBytes;
  const size_t T = d->T, E = d->E, K = d->topk, H = d->H;
  const size_t nblk = moe::route_blocks(d->T);
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += up(bytes);
    return at;
  };
  if (which == MOE_WS_ROUTE || which == MOE_WS_PERMUTE ||
      which == MOE_WS_FORWARD) {
    L.block_counts = take(nblk * E * 4);
    L.block_base = take(nblk * E * 4);
  }
  if (which == MOE_WS_PERMUTE) L.counts = take(E * 4);
  if (which == MOE_WS_EXPERT_BWD) {
    const size_t cap = moe::expert_backward_rows_cap(d->T, d->topk, d->E);
    const size_t I = d->I, Is = d->I_shared;
    const size_t nfb = (I + 255) / 256;
    L.block_counts = take(nblk * E * 4);
    L.block_base = take(nblk * E * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.dest = take(T * K * 4);
    L.src_row = take(T * K * 4);
    L.b_poff = take((E + 1) * 4);
    L.b_ticket = take(4);
    L.b_pdest = take(T * K * 4);
    L.b_gp = take(cap * 4);
    L.b_xpp = take(cap * H * 2);
    L.b_dpp = take(cap * H * 2);
    L.b_p = take(cap * I * 4);
    L.b_q = take(cap * I * 4);
    L.b_hg = take(cap * I * 2);
    L.b_dp = take(cap * I * 2);
    L.b_dq = take(cap * I * 2);
    L.b_dgp = take(cap * nfb * 4);
    L.b_dxpp = take(cap * H * 2);
    L.b_ps = take(T * Is * 4);
    L.b_qs = take(T * Is * 4);
    L.b_hgs = take(T * Is * 2);
    L.b_dps = take(T * Is * 2);
    L.b_dqs = take(T * Is * 2);
    L.b_dxs = take(T * H * 2);
  }
  if (which == MOE_WS_FORWARD) {
    L.logits = take(T * E * 4);
    L.idx = take(T * K * 4);
    L.gate = take(T * K * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.dest = take(T * K * 4);
    L.src_row = take(T * K * 4);
    if (!gather_rows(d)) L.xp = take(T * K * H * 2);
    L.yp = take(T * K * H * 2);
    L.ys = take(T * H * 2);
  }
  if (which == MOE_WS_EXPERT_FFN || which == MOE_WS_FORWARD) {
    L.h = take(T * K * (size_t)d->I * 2);
    L.hs = take(T * (size_t)d->I_shared * 2);
  }
  if (which == MOE_WS_ROUTER_LOGITS || which == MOE_WS_FORWARD) {
    L.w_split = take(3 * E * H * 2);
    const size_t ks = moe::router_ksplit(d->T, d->H, d->E);
    if (ks > 1) L.r_partial = take(ks * T * E * 4);
  }
  if (which == MOE_WS_SEQ_BALANCE) {
    L.bal_sp = take(T * E * 4);
    L.bal_flags = take(T * E);
    L.bal_pP = take(moe::kBalPartialElems * 4);
    L.bal_pc = take(moe::kBalPartialElems * 4);
  }
  if (which == MOE_WS_EXPERT_FFN_FP8) {
    const size_t I = d->I, Is = d->I_shared;
    L.f8_mq = take(T * K * I);
    L.f8_ms = take(T * K * (I / 128) * 4);
    L.f8_msq = take(T * Is);
    L.f8_mss = take(T * (Is / 128) * 4);
  }
  if (which == MOE_WS_EXPERT_FFN_MX) {
    const size_t I = d->I, Is = d->I_shared;
    L.mx_mq = take(T * K * I);
    L.mx_ms = take(T * K * (I / 128));
    L.mx_msq = take(T * Is);
    L.mx_mss = take(T * (Is / 128));
  }
  L.total = o;
  // one MOE_WS_FORWARD workspace serves every entry point
  if (which == MOE_WS_FORWARD) {
    L.total = std::max(L.total, layout(d, MOE_WS_SEQ_BALANCE).total);
    L.total = std::max(L.total, layout(d, MOE_WS_EXPERT_FFN_FP8).total);
    L.total = std::max(L.total, layout(d, MOE_WS_EXPERT_FFN_MX).total);
  }
  return L;
}

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

moe_status_t check_ws(const moe_dims_t* d, moe_ws_kind_t which, void* ws,
                      size_t ws_bytes) {
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_ALIGNMENT;
  if (ws_bytes < layout(d, which).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

inline moe_status_t cuda_ok(cudaError_t e) {
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

#define MOE_TRY(expr)                      \
  do {                                     \
    const moe_status_t st_ = (expr);       \
    if (st_ != MOE_OK) return st_;         \
  } while (0)

#define MOE_NEED(p) \
  do {              \
    if ((p) == nullptr) return MOE_ERR_INVALID_ARG; \
  } while (0)

// a [T, ...] tensor may be NULL when there are no tokens
#define MOE_NEED_T(p) \
  do {                \
    if (d->T > 0 && (p) == nullptr) return MOE_ERR_INVALID_ARG; \
  } while (0)

#define MOE_ALIGN(p) \
  do {               \
    if ((p) != nullptr && !aligned16(p)) return MOE_ERR_ALIGNMENT; \
  } while (0)

moe_status_t check_weights(const moe_weights_t* w) {
  MOE_NEED(w);
  MOE_NEED(w->w_router);
  MOE_NEED(w->w1);
  MOE_NEED(w->w3);
  MOE_NEED(w->w2);
  MOE_NEED(w->ws1);
  MOE_NEED(w->ws3);
  MOE_NEED(w->ws2);
  MOE_ALIGN(w->w_router);
  MOE_ALIGN(w->router_offset);
  MOE_ALIGN(w->router_split);
  MOE_ALIGN(w->w1);
  MOE_ALIGN(w->w3);
  MOE_ALIGN(w->w2);
  MOE_ALIGN(w->ws1);
  MOE_ALIGN(w->ws3);
  MOE_ALIGN(w->ws2);
  return MOE_OK;
}

moe_status_t ffn_launch(const moe_dims_t* d, const moe_weights_t* w,
                        const uint16_t* xp, const uint16_t* x,
                        const int32_t* offsets, uint16_t* h, uint16_t* hs,
                        uint16_t* yp, uint16_t* ys, DevStatus* st,
                        cudaStream_t s, void* between_event = nullptr,
                        const int32_t* src_row = nullptr) {
  moe::FfnArgs a;
  a.T = d->T;
  a.H = d->H;
  a.E = d->E;
  a.topk = d->topk;
  a.I = d->I;
  a.I_shared = d->I_shared;
  a.xp = xp;
  a.x = x;
  a.src_row = src_row;
  a.offsets = offsets;
  a.w1 = w->w1;
  a.w3 = w->w3;
  a.w2 = w->w2;
  a.ws1 = w->ws1;
  a.ws3 = w->ws3;
  a.ws2 = w->ws2;
  a.h = h;
  a.hs = hs;
  a.yp = yp;
  a.ys = ys;
  a.status = st;
  a.wait_limit_ns = g_wait_limit_ns;
  a.between_event = between_event;
  return static_cast<moe_status_t>(moe::launch_expert_ffn(a, s));
}

// z = x W_r^T (+ offset): tensor cores (exact bf16 split of W_r) when
// E % 16 == 0, else the fp32 SIMT kernel
// (presplit: the caller's moe_router_weight_split of w_router, or NULL:
// split into w_split now)
moe_status_t router_logits_launch(const moe_dims_t* d, const uint16_t* x,
                                  const float* w_router,
                                  const float* offset, float* logits,
                                  uint16_t* w_split, float* partial,
                                  DevStatus* st, cudaStream_t s,
                                  const uint16_t* presplit = nullptr) {
  if (moe::router_tile_n(d->T, d->E) == 0)
    return cuda_ok(moe::launch_router_logits(x, w_router, offset, logits,
                                             d->T, d->H, d->E, s));
  if (presplit == nullptr)
    MOE_TRY(cuda_ok(moe::launch_split_router_weight(w_router, d->E, d->H,
                                                    w_split, s)));
  return static_cast<moe_status_t>(moe::launch_router_logits_tc(
      x, presplit ? presplit : w_split, offset, logits, partial, d->T, d->H,
      d->E, st, g_wait_limit_ns, s));
}

}  // namespace

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

moe_status_t moe_router_weight_split(const float* w_router, int32_t E,
                                     int32_t H, uint16_t* split,
                                     moe_stream_t stream) {
  if (E <= 0 || H <= 0) return MOE_ERR_INVALID_ARG;
  if (E % 16 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_NEED(w_router);
  MOE_NEED(split);
  MOE_ALIGN(w_router);
  MOE_ALIGN(split);
  return cuda_ok(
      moe::launch_split_router_weight(w_router, E, H, split, cs(stream)));
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_ALIGNMENT: return "MOE_ERR_ALIGNMENT";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS";
  }
  return "MOE_ERR_UNKNOWN";
}

void moe_set_profile_events(void* const* events, int32_t n) {
  g_prof_events = (events != nullptr && n >= MOE_FORWARD_KERNELS + 1)
                      ? events
                      : nullptr;
}

void moe_set_gemm_ctas(int32_t n) { moe::set_gemm_ctas(n); }

void moe_set_wait_timeout_ns(uint64_t ns) {
  g_wait_limit_ns = ns == 0 ? kDefaultWaitNs : ns;
}

size_t moe_workspace_bytes(const moe_dims_t* d, moe_ws_kind_t which) {
  const bool ffn = which == MOE_WS_EXPERT_FFN || which == MOE_WS_FORWARD ||
                   which == MOE_WS_EXPERT_FFN_FP8 ||
                   which == MOE_WS_EXPERT_BWD ||
                   which == MOE_WS_EXPERT_FFN_MX;
  if (which < MOE_WS_ROUTE || which > MOE_WS_EXPERT_FFN_MX) return 0;
  // the expert GEMMs alone (moe_expert_ffn, moe_expert_ffn_routed and
  // their FP8 power-of-two forms) do not route: their workspace takes any
  // expert count
  if (which == MOE_WS_EXPERT_FFN || which == MOE_WS_EXPERT_FFN_MX) {
    if (check_ffn_only_dims(d) != MOE_OK) return 0;
  } else if (check_dims(d, ffn) != MOE_OK) {
    return 0;
  }
  return layout(d, which).total;
}

moe_status_t moe_get_device_error(void* ws, moe_stream_t stream) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  DevStatus h{0, 0};
  if (cudaStreamSynchronize(cs(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (h.code != 0) {
    const DevStatus zero{0, 0};
    if (cudaMemcpy(ws, &zero, sizeof(zero), cudaMemcpyHostToDevice) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return static_cast<moe_status_t>(h.code);
}

moe_status_t moe_router_logits(const moe_dims_t* d, const uint16_t* x,
                               const float* w_router,
                               const float* router_offset, float* logits,
                               void* ws, size_t ws_bytes,
                               moe_stream_t stream) {
  MOE_TRY(check_dims(d, false));
  MOE_NEED_T(x);
  MOE_NEED(w_router);
  MOE_NEED_T(logits);
  MOE_ALIGN(x);
  MOE_ALIGN(w_router);
  MOE_ALIGN(router_offset);
  MOE_ALIGN(logits);
  MOE_TRY(check_ws(d, MOE_WS_ROUTER_LOGITS, ws, ws_bytes));
  if (d->T == 0) return MOE_OK;
  const Layout L = layout(d, MOE_WS_ROUTER_LOGITS);
  return router_logits_launch(
      d, x, w_router, router_offset, logits, at<uint16_t>(ws, L.w_split),
      L.r_partial ? at<float>(ws, L.r_partial) : nullptr,
      at<DevStatus>(ws, 0), cs(stream));
}

moe_status_t moe_route(const moe_dims_t* d, const float* logits,
                       const float* bias, int32_t* topk_idx, float* topk_gate,
                       int32_t* counts, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  MOE_TRY(check_dims(d, false));
  MOE_NEED_T(logits);
  MOE_NEED(bias);
  MOE_NEED_T(topk_idx);
  MOE_NEED_T(topk_gate);
  MOE_NEED(counts);
  MOE_ALIGN(logits);
  MOE_ALIGN(bias);
  MOE_ALIGN(topk_idx);
  MOE_ALIGN(topk_gate);
  MOE_ALIGN(counts);
  MOE_TRY(check_ws(d, MOE_WS_ROUTE, ws, ws_bytes));
  const Layout L = layout(d, MOE_WS_ROUTE);
  cudaStream_t s = cs(stream);
  if (d->T == 0) {
    return cuda_ok(cudaMemsetAsync(counts, 0, sizeof(int32_t) * d->E, s));
  }
  int32_t* bc = at<int32_t>(ws, L.block_counts);
  MOE_TRY(cuda_ok(moe::launch_route(logits, bias, d->T, d->E, d->n_group,
                                    d->topk_group, d->topk, topk_idx,
                                    topk_gate, bc, s)));
  return cuda_ok(moe::launch_scan(bc, d->T, d->E, d->topk, counts, nullptr,
                                  nullptr, 0.f, s));
}

moe_status_t moe_permute(const moe_dims_t* d, const uint16_t* x,
                         const int32_t* topk_idx, int32_t* offsets,
                         int32_t* dest, int32_t* src_row, uint16_t* xp,
                         void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_dims(d, false));
  MOE_NEED_T(topk_idx);
  MOE_NEED(offsets);
  MOE_NEED_T(dest);
  MOE_NEED_T(src_row);
  if (xp != nullptr) MOE_NEED_T(x);
  MOE_ALIGN(x);
  MOE_ALIGN(topk_idx);
  MOE_ALIGN(offsets);
  MOE_ALIGN(dest);
  MOE_ALIGN(src_row);
  MOE_ALIGN(xp);
  MOE_TRY(check_ws(d, MOE_WS_PERMUTE, ws, ws_bytes));
  const Layout L = layout(d, MOE_WS_PERMUTE);
  cudaStream_t s = cs(stream);
  if (d->T == 0)
    return cuda_ok(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (d->E + 1), s));
  DevStatus* st = at<DevStatus>(ws, 0);
  int32_t* bc = at<int32_t>(ws, L.block_counts);
  int32_t* bb = at<int32_t>(ws, L.block_base);
  int32_t* cnt = at<int32_t>(ws, L.counts);
  MOE_TRY(cuda_ok(moe::launch_block_counts(topk_idx, d->T, d->E, d->topk, bc,
                                           st, s)));
  MOE_TRY(cuda_ok(moe::launch_scan(bc, d->T, d->E, d->topk, cnt, bb, nullptr,
                                   0.f, s)));
  MOE_TRY(cuda_ok(moe::launch_dest(topk_idx, cnt, bb, d->T, d->E, d->topk,
                                   offsets, dest, src_row, nullptr, st, s)));
  if (xp != nullptr)
    MOE_TRY(cuda_ok(moe::launch_gather(x, dest, d->T, d->H, d->topk, xp, s)));
  return MOE_OK;
}

moe_status_t moe_expert_ffn(const moe_dims_t* d, const moe_weights_t* w,
                            const uint16_t* xp, const uint16_t* x,
                            const int32_t* offsets, uint16_t* yp,
                            uint16_t* ys, void* ws, size_t ws_bytes,
                            moe_stream_t stream) {
  MOE_TRY(check_dims(d, true));
  MOE_TRY(check_weights(w));
  MOE_NEED_T(xp);
  MOE_NEED_T(x);
  MOE_NEED(offsets);
  MOE_NEED_T(yp);
  MOE_NEED_T(ys);
  MOE_ALIGN(xp);
  MOE_ALIGN(x);
  MOE_ALIGN(offsets);
  MOE_ALIGN(yp);
  MOE_ALIGN(ys);
  MOE_TRY(check_ws(d, MOE_WS_EXPERT_FFN, ws, ws_bytes));
  if (d->T == 0) return MOE_OK;
  const Layout L = layout(d, MOE_WS_EXPERT_FFN);
  return ffn_launch(d, w, xp, x, offsets, at<uint16_t>(ws, L.h),
                    at<uint16_t>(ws, L.hs), yp, ys, at<DevStatus>(ws, 0),
                    cs(stream));
}

moe_status_t moe_expert_ffn_routed(const moe_dims_t* d, const moe_weights_t* w,
                                   const uint16_t* xp, const int32_t* offsets,
                                   uint16_t* yp, void* ws, size_t ws_bytes,
                                   moe_stream_t stream) {
  MOE_TRY(check_ffn_only_dims(d));
  MOE_NEED(w);
  MOE_NEED(w->w1);
  MOE_NEED(w->w3);
  MOE_NEED(w->w2);
  MOE_ALIGN(w->w1);
  MOE_ALIGN(w->w3);
  MOE_ALIGN(w->w2);
  MOE_NEED_T(xp);
  MOE_NEED(offsets);
  MOE_NEED_T(yp);
  MOE_ALIGN(xp);
  MOE_ALIGN(offsets);
  MOE_ALIGN(yp);
  MOE_TRY(check_ws(d, MOE_WS_EXPERT_FFN, ws, ws_bytes));
  if (d->T == 0) return MOE_OK;
  const Layout L = layout(d, MOE_WS_EXPERT_FFN);
  moe_weights_t rw = *w;
  rw.ws1 = rw.ws3 = rw.ws2 = nullptr;
  return ffn_launch(d, &rw, xp, nullptr, offsets, at<uint16_t>(ws, L.h),
                    nullptr, yp, nullptr, at<DevStatus>(ws, 0), cs(stream));
}

moe_status_t moe_ep_plan(int32_t n_src, int32_t n_local, const int32_t* counts,
                         int64_t rows, int32_t* perm, int32_t* offsets_local,
                         void* ws, moe_stream_t stream) {
  if (n_src < 1 || n_local < 1 || rows < 0 || rows >= (1ll << 31))
    return MOE_ERR_INVALID_ARG;
  if ((long long)n_src * n_local > moe::ep_plan_max_cells())
    return MOE_ERR_UNSUPPORTED;
  MOE_NEED(counts);
  MOE_NEED(offsets_local);
  if (rows > 0) MOE_NEED(perm);
  MOE_ALIGN(counts);
  MOE_ALIGN(perm);
  MOE_ALIGN(offsets_local);
  MOE_ALIGN(ws);
  return cuda_ok(moe::launch_ep_plan(
      counts, n_src, n_local, rows, perm, offsets_local,
      ws ? at<DevStatus>(ws, 0) : nullptr, cs(stream)));
}

moe_status_t moe_ep_permute_rows(const void* in, int64_t rows,
                                 int64_t row_bytes, const int32_t* perm,
                                 int32_t inverse, void* out, void* ws,
                                 moe_stream_t stream) {
  if (rows < 0 || rows >= (1ll << 31) || row_bytes <= 0)
    return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  MOE_NEED(in);
  MOE_NEED(out);
  MOE_NEED(perm);
  MOE_ALIGN(in);
  MOE_ALIGN(out);
  MOE_ALIGN(perm);
  MOE_ALIGN(ws);
  return cuda_ok(moe::launch_ep_rows(in, rows, row_bytes, perm,
                                     inverse ? 1 : 0, out,
                                     ws ? at<DevStatus>(ws, 0) : nullptr,
                                     cs(stream)));
}

moe_status_t moe_combine(const moe_dims_t* d, const uint16_t* x,
                         const uint16_t* ys, const uint16_t* yp,
                         const int32_t* dest, const float* topk_gate,
                         uint16_t* out, moe_stream_t stream) {
  MOE_TRY(check_dims(d, false));
  MOE_NEED_T(x);
  MOE_NEED_T(ys);
  MOE_NEED_T(yp);
  MOE_NEED_T(dest);
  MOE_NEED_T(topk_gate);
  MOE_NEED_T(out);
  MOE_ALIGN(x);
  MOE_ALIGN(ys);
  MOE_ALIGN(yp);
  MOE_ALIGN(dest);
  MOE_ALIGN(topk_gate);
  MOE_ALIGN(out);
  if (d->T == 0) return MOE_OK;
  return cuda_ok(moe::launch_combine(x, ys, yp, dest, topk_gate, d->T, d->H,
                                     d->topk, out, cs(stream)));
}

moe_status_t moe_seq_balance_loss(const moe_dims_t* d, const float* logits,
                                  int32_t seq_len, float alpha,
                                  int32_t* counts_seq, float* P_seq,
                                  float* loss, void* ws, size_t ws_bytes,
                                  moe_stream_t stream) {
  MOE_TRY(check_dims(d, false));
  if (seq_len < 1 || !std::isfinite(alpha)) return MOE_ERR_INVALID_ARG;
  MOE_NEED_T(logits);
  MOE_NEED_T(counts_seq);
  MOE_NEED_T(P_seq);
  MOE_NEED_T(loss);
  MOE_ALIGN(logits);
  MOE_ALIGN(counts_seq);
  MOE_ALIGN(P_seq);
  MOE_ALIGN(loss);
  MOE_TRY(check_ws(d, MOE_WS_SEQ_BALANCE, ws, ws_bytes));
  if (d->T == 0) return MOE_OK;
  const Layout L = layout(d, MOE_WS_SEQ_BALANCE);
  const long long n_seq = ((long long)d->T + seq_len - 1) / seq_len;
  const int rs = moe::seq_balance_splits(d->T, d->E, seq_len);
  if (rs > 1 && n_seq * rs * d->E > moe::kBalPartialElems)
    return MOE_ERR_UNSUPPORTED;  // cannot happen: the split rule bounds it
  return cuda_ok(moe::launch_seq_balance(
      logits, d->T, d->E, d->topk, seq_len, alpha, at<float>(ws, L.bal_sp),
      at<uint8_t>(ws, L.bal_flags), P_seq, counts_seq,
      at<float>(ws, L.bal_pP), at<int32_t>(ws, L.bal_pc), loss, cs(stream)));
}

moe_status_t moe_quantize_fp8_blocks(const uint16_t* w, int64_t rows,
                                     int64_t cols, uint8_t* q, float* scale,
                                     moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || rows % 128 != 0 || cols % 128 != 0)
    return MOE_ERR_INVALID_ARG;
  if (rows / 128 > 65535 || cols > (1 << 30)) return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  MOE_NEED(w);
  MOE_NEED(q);
  MOE_NEED(scale);
  MOE_ALIGN(w);
  MOE_ALIGN(q);
  MOE_ALIGN(scale);
  return cuda_ok(
      moe::launch_quant_blocks(w, rows, (int)cols, q, scale, cs(stream)));
}

moe_status_t moe_quantize_fp8_rows(const uint16_t* x, int64_t rows,
                                   int64_t cols, uint8_t* q, float* scale,
                                   moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (cols > (1 << 30) || rows * (cols / 128) >= (1ll << 40))
    return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  MOE_NEED(x);
  MOE_NEED(q);
  MOE_NEED(scale);
  MOE_ALIGN(x);
  MOE_ALIGN(q);
  MOE_ALIGN(scale);
  return cuda_ok(moe::launch_quant_rows(x, rows, (int)cols, nullptr, 0, q,
                                        scale, nullptr, nullptr, nullptr,
                                        cs(stream)));
}

moe_status_t moe_permute_fp8(const moe_dims_t* d, const uint16_t* x,
                             const int32_t* dest, uint8_t* xq, float* xs,
                             uint8_t* xpq, float* xps, void* ws,
                             size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_dims(d, false));
  if (d->H % 128 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_NEED_T(x);
  MOE_NEED_T(dest);
  MOE_NEED_T(xq);
  MOE_NEED_T(xs);
  MOE_NEED_T(xpq);
  MOE_NEED_T(xps);
  MOE_ALIGN(x);
  MOE_ALIGN(dest);
  MOE_ALIGN(xq);
  MOE_ALIGN(xs);
  MOE_ALIGN(xpq);
  MOE_ALIGN(xps);
  MOE_TRY(check_ws(d, MOE_WS_PERMUTE, ws, ws_bytes));
  if (d->T == 0) return MOE_OK;
  return cuda_ok(moe::launch_quant_rows(
      x, d->T, d->H, dest, d->topk, xq, xs, xpq, xps,
      at<DevStatus>(ws, 0), cs(stream)));
}

moe_status_t moe_expert_ffn_fp8(const moe_dims_t* d, const moe_weights_fp8_t* w,
                                const uint8_t* xpq, const float* xps,
                                const uint8_t* xq, const float* xs,
                                const int32_t* offsets, uint16_t* yp,
                                uint16_t* ys, void* ws, size_t ws_bytes,
                                moe_stream_t stream) {
  MOE_TRY(check_dims(d, true));
  if (!moe::fp8_ffn_supported(d->H, d->I, d->I_shared, d->E))
    return MOE_ERR_UNSUPPORTED;
  MOE_NEED(w);
  const void* wp[12] = {w->w1,  w->w1_scale,  w->w3,  w->w3_scale,
                        w->w2,  w->w2_scale,  w->ws1, w->ws1_scale,
                        w->ws3, w->ws3_scale, w->ws2, w->ws2_scale};
  for (const void* ptr : wp) {
    MOE_NEED(ptr);
    MOE_ALIGN(ptr);
  }
  MOE_NEED_T(xpq);
  MOE_NEED_T(xps);
  MOE_NEED_T(xq);
  MOE_NEED_T(xs);
  MOE_NEED(offsets);
  MOE_NEED_T(yp);
  MOE_NEED_T(ys);
  MOE_ALIGN(xpq);
  MOE_ALIGN(xps);
  MOE_ALIGN(xq);
  MOE_ALIGN(xs);
  MOE_ALIGN(offsets);
  MOE_ALIGN(yp);
  MOE_ALIGN(ys);
  MOE_TRY(check_ws(d, MOE_WS_EXPERT_FFN_FP8, ws, ws_bytes));
  if (d->T == 0) return MOE_OK;
  const Layout L = layout(d, MOE_WS_EXPERT_FFN_FP8);
  moe::FfnFp8Args a;
  a.T = d->T;
  a.H = d->H;
  a.E = d->E;
  a.topk = d->topk;
  a.I = d->I;
  a.I_shared = d->I_shared;
  a.xpq = xpq;
  a.xq = xq;
  a.xps = xps;
  a.xs = xs;
  a.offsets = offsets;
  a.w1 = w->w1;
  a.w3 = w->w3;
  a.w2 = w->w2;
  a.w1s = w->w1_scale;
  a.w3s = w->w3_scale;
  a.w2s = w->w2_scale;
  a.ws1 = w->ws1;
  a.ws3 = w->ws3;
  a.ws2 = w->ws2;
  a.ws1s = w->ws1_scale;
  a.ws3s = w->ws3_scale;
  a.ws2s = w->ws2_scale;
  a.mq = at<uint8_t>(ws, L.f8_mq);
  a.ms = at<float>(ws, L.f8_ms);
  a.msq = at<uint8_t>(ws, L.f8_msq);
  a.mss = at<float>(ws, L.f8_mss);
  a.yp = yp;
  a.ys = ys;
  a.status = at<DevStatus>(ws, 0);
  a.wait_limit_ns = g_wait_limit_ns;
  const int rc = moe::launch_expert_ffn_fp8(a, cs(stream));
  return static_cast<moe_status_t>(rc);
}

moe_status_t moe_quantize_mx_blocks(const uint16_t* w, int64_t rows,
                                    int64_t cols, uint8_t* q, uint8_t* scale,
                                    moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || rows % 128 != 0 || cols % 128 != 0)
    return MOE_ERR_INVALID_ARG;
  if (rows / 128 > 65535 || cols > (1 << 30)) return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  MOE_NEED(w);
  MOE_NEED(q);
  MOE_NEED(scale);
  MOE_ALIGN(w);
  MOE_ALIGN(q);
  MOE_ALIGN(scale);
  return cuda_ok(
      moe::launch_quant_blocks_e8(w, rows, (int)cols, q, scale, cs(stream)));
}

moe_status_t moe_quantize_mx_rows(const uint16_t* x, int64_t rows,
                                  int64_t cols, uint8_t* q, uint8_t* scale,
                                  moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (cols > (1 << 30) || rows * (cols / 128) >= (1ll << 40))
    return MOE_ERR_UNSUPPORTED;
  if (rows == 0) return MOE_OK;
  MOE_NEED(x);
  MOE_NEED(q);
  MOE_NEED(scale);
  MOE_ALIGN(x);
  MOE_ALIGN(q);
  MOE_ALIGN(scale);
  return cuda_ok(moe::launch_quant_rows_e8(x, rows, (int)cols, nullptr, 0, q,
                                           scale, nullptr, nullptr, nullptr,
                                           cs(stream)));
}

moe_status_t moe_permute_mx(const moe_dims_t* d, const uint16_t* x,
                            const int32_t* dest, uint8_t* xq, uint8_t* xs,
                            uint8_t* xpq, uint8_t* xps, void* ws,
                            size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_dims(d, false));
  if (d->H % 128 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_NEED_T(x);
  MOE_NEED_T(dest);
  MOE_NEED_T(xq);
  MOE_NEED_T(xs);
  MOE_NEED_T(xpq);
  MOE_NEED_T(xps);
  MOE_ALIGN(x);
  MOE_ALIGN(dest);
  MOE_ALIGN(xq);
  MOE_ALIGN(xs);
  MOE_ALIGN(xpq);
  MOE_ALIGN(xps);
  MOE_TRY(check_ws(d, MOE_WS_PERMUTE, ws, ws_bytes));
  if (d->T == 0) return MOE_OK;
  return cuda_ok(moe::launch_quant_rows_e8(
      x, d->T, d->H, dest, d->topk, xq, xs, xpq, xps,
      at<DevStatus>(ws, 0), cs(stream)));
}

moe_status_t moe_expert_ffn_mx(const moe_dims_t* d, const moe_weights_mx_t* w,
                               const uint8_t* xpq, const uint8_t* xps,
                               const uint8_t* xq, const uint8_t* xs,
                               const int32_t* offsets, uint16_t* yp,
                               uint16_t* ys, void* ws, size_t ws_bytes,
                               moe_stream_t stream) {
  MOE_TRY(check_dims(d, true));
  if (!moe::mx_ffn_supported(d->H, d->I, d->I_shared, d->E))
    return MOE_ERR_UNSUPPORTED;
  MOE_NEED(w);
  const void* wp[12] = {w->w1,  w->w1_scale,  w->w3,  w->w3_scale,
                        w->w2,  w->w2_scale,  w->ws1, w->ws1_scale,
                        w->ws3, w->ws3_scale, w->ws2, w->ws2_scale};
  for (const void* ptr : wp) {
    MOE_NEED(ptr);
    MOE_ALIGN(ptr);
  }
  MOE_NEED_T(xpq);
  MOE_NEED_T(xps);
  MOE_NEED_T(xq);
  MOE_NEED_T(xs);
  MOE_NEED(offsets);
  MOE_NEED_T(yp);
  MOE_NEED_T(ys);
  MOE_ALIGN(xpq);
  MOE_ALIGN(xps);
  MOE_ALIGN(xq);
  MOE_ALIGN(xs);
  MOE_ALIGN(offsets);
  MOE_ALIGN(yp);
  MOE_ALIGN(ys);
  MOE_TRY(check_ws(d, MOE_WS_EXPERT_FFN_MX, ws, ws_bytes));
  if (d->T == 0) return MOE_OK;
  const Layout L = layout(d, MOE_WS_EXPERT_FFN_MX);
  moe::FfnMxArgs a;
  a.T = d->T;
  a.H = d->H;
  a.E = d->E;
  a.topk = d->topk;
  a.I = d->I;
  a.I_shared = d->I_shared;
  a.xpq = xpq;
  a.xq = xq;
  a.xps = xps;
  a.xs = xs;
  a.offsets = offsets;
  a.w1 = w->w1;
  a.w3 = w->w3;
  a.w2 = w->w2;
  a.w1s = w->w1_scale;
  a.w3s = w->w3_scale;
  a.w2s = w->w2_scale;
  a.ws1 = w->ws1;
  a.ws3 = w->ws3;
  a.ws2 = w->ws2;
  a.ws1s = w->ws1_scale;
  a.ws3s = w->ws3_scale;
  a.ws2s = w->ws2_scale;
  a.mq = at<uint8_t>(ws, L.mx_mq);
  a.ms = at<uint8_t>(ws, L.mx_ms);
  a.msq = at<uint8_t>(ws, L.mx_msq);
  a.mss = at<uint8_t>(ws, L.mx_mss);
  a.yp = yp;
  a.ys = ys;
  a.status = at<DevStatus>(ws, 0);
  a.wait_limit_ns = g_wait_limit_ns;
  const int rc = moe::launch_expert_ffn_mx(a, cs(stream));
  return static_cast<moe_status_t>(rc);
}

moe_status_t moe_expert_ffn_mx_routed(const moe_dims_t* d,
                                      const moe_weights_mx_t* w,
                                      const uint8_t* xpq, const uint8_t* xps,
                                      const int32_t* offsets, uint16_t* yp,
                                      void* ws, size_t ws_bytes,
                                      moe_stream_t stream) {
  MOE_TRY(check_ffn_only_dims(d));
  if (!moe::mx_ffn_supported(d->H, d->I, d->I_shared, d->E))
    return MOE_ERR_UNSUPPORTED;
  MOE_NEED(w);
  const void* wp[6] = {w->w1, w->w1_scale, w->w3, w->w3_scale, w->w2,
                       w->w2_scale};
  for (const void* ptr : wp) {
    MOE_NEED(ptr);
    MOE_ALIGN(ptr);
  }
  MOE_NEED_T(xpq);
  MOE_NEED_T(xps);
  MOE_NEED(offsets);
  MOE_NEED_T(yp);
  MOE_ALIGN(xpq);
  MOE_ALIGN(xps);
  MOE_ALIGN(offsets);
  MOE_ALIGN(yp);
  MOE_TRY(check_ws(d, MOE_WS_EXPERT_FFN_MX, ws, ws_bytes));
  if (d->T == 0) return MOE_OK;
  const Layout L = layout(d, MOE_WS_EXPERT_FFN_MX);
  moe::FfnMxArgs a;
  std::memset(&a, 0, sizeof(a));
  a.T = d->T;
  a.H = d->H;
  a.E = d->E;
  a.topk = d->topk;
  a.I = d->I;
  a.I_shared = d->I_shared;
  a.xpq = xpq;
  a.xps = xps;
  a.offsets = offsets;
  a.w1 = w->w1;
  a.w3 = w->w3;
  a.w2 = w->w2;
  a.w1s = w->w1_scale;
  a.w3s = w->w3_scale;
  a.w2s = w->w2_scale;
  a.mq = at<uint8_t>(ws, L.mx_mq);
  a.ms = at<uint8_t>(ws, L.mx_ms);
  a.yp = yp;
  a.status = at<DevStatus>(ws, 0);
  a.wait_limit_ns = g_wait_limit_ns;
  return static_cast<moe_status_t>(moe::launch_expert_ffn_mx(a, cs(stream)));
}

moe_status_t moe_expert_backward(const moe_dims_t* d, const moe_weights_t* w,
                                 const uint16_t* x, const uint16_t* dout,
                                 const int32_t* topk_idx,
                                 const float* topk_gate, int accumulate,
                                 uint16_t* dx, float* dgate, float* dw1,
                                 float* dw3, float* dw2, float* dws1,
                                 float* dws3, float* dws2, void* ws,
                                 size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_dims(d, true));
  MOE_NEED(w);
  MOE_NEED(w->w1);
  MOE_NEED(w->w3);
  MOE_NEED(w->w2);
  MOE_NEED(w->ws1);
  MOE_NEED(w->ws3);
  MOE_NEED(w->ws2);
  MOE_ALIGN(w->w1);
  MOE_ALIGN(w->w3);
  MOE_ALIGN(w->w2);
  MOE_ALIGN(w->ws1);
  MOE_ALIGN(w->ws3);
  MOE_ALIGN(w->ws2);
  MOE_NEED_T(x);
  MOE_NEED_T(dout);
  MOE_NEED_T(topk_idx);
  MOE_NEED_T(topk_gate);
  MOE_NEED_T(dx);
  MOE_NEED_T(dgate);
  MOE_NEED(dw1);
  MOE_NEED(dw3);
  MOE_NEED(dw2);
  MOE_NEED(dws1);
  MOE_NEED(dws3);
  MOE_NEED(dws2);
  const void* al[] = {x, dout, topk_idx, topk_gate, dx, dgate,
                      dw1, dw3, dw2, dws1, dws3, dws2};
  for (const void* q : al) MOE_ALIGN(q);
  MOE_TRY(check_ws(d, MOE_WS_EXPERT_BWD, ws, ws_bytes));
  cudaStream_t s = cs(stream);
  const size_t E = d->E, H = d->H, I = d->I, Is = d->I_shared;
  if (d->T == 0) {
    if (!accumulate) {
      // no tokens: every weight gradient is zero
      MOE_TRY(cuda_ok(cudaMemsetAsync(dw1, 0, E * I * H * 4, s)));
      MOE_TRY(cuda_ok(cudaMemsetAsync(dw3, 0, E * I * H * 4, s)));
      MOE_TRY(cuda_ok(cudaMemsetAsync(dw2, 0, E * H * I * 4, s)));
      MOE_TRY(cuda_ok(cudaMemsetAsync(dws1, 0, Is * H * 4, s)));
      MOE_TRY(cuda_ok(cudaMemsetAsync(dws3, 0, Is * H * 4, s)));
      MOE_TRY(cuda_ok(cudaMemsetAsync(dws2, 0, H * Is * 4, s)));
    }
    return MOE_OK;
  }
  const Layout L = layout(d, MOE_WS_EXPERT_BWD);
  DevStatus* st = at<DevStatus>(ws, 0);
  int32_t* bc = at<int32_t>(ws, L.block_counts);
  int32_t* bb = at<int32_t>(ws, L.block_base);
  int32_t* cnt = at<int32_t>(ws, L.counts);
  int32_t* off = at<int32_t>(ws, L.offsets);
  int32_t* dst = at<int32_t>(ws, L.dest);
  int32_t* src = at<int32_t>(ws, L.src_row);
  const int T = d->T, K = d->topk;
  MOE_TRY(cuda_ok(moe::launch_block_counts(topk_idx, T, d->E, K, bc, st, s)));
  MOE_TRY(cuda_ok(moe::launch_scan(bc, T, d->E, K, cnt, bb, nullptr, 0.f, s)));
  MOE_TRY(cuda_ok(moe::launch_dest(topk_idx, cnt, bb, T, d->E, K, off, dst,
                                   src, nullptr, st, s)));
  moe::BwdArgs a;
  a.T = T;
  a.H = d->H;
  a.E = d->E;
  a.topk = K;
  a.I = d->I;
  a.I_shared = d->I_shared;
  a.x = x;
  a.dout = dout;
  a.topk_idx = topk_idx;
  a.dest = dst;
  a.offsets = off;
  a.counts = cnt;
  a.gate = topk_gate;
  a.w1 = w->w1;
  a.w3 = w->w3;
  a.w2 = w->w2;
  a.ws1 = w->ws1;
  a.ws3 = w->ws3;
  a.ws2 = w->ws2;
  a.poff = at<int32_t>(ws, L.b_poff);
  a.ticket = at<int>(ws, L.b_ticket);
  a.pdest = at<int32_t>(ws, L.b_pdest);
  a.gp = at<float>(ws, L.b_gp);
  a.xpp = at<uint16_t>(ws, L.b_xpp);
  a.dpp = at<uint16_t>(ws, L.b_dpp);
  a.p_r = at<float>(ws, L.b_p);
  a.q_r = at<float>(ws, L.b_q);
  a.hg_r = at<uint16_t>(ws, L.b_hg);
  a.dp_r = at<uint16_t>(ws, L.b_dp);
  a.dq_r = at<uint16_t>(ws, L.b_dq);
  a.dgp = at<float>(ws, L.b_dgp);
  a.dxpp = at<uint16_t>(ws, L.b_dxpp);
  a.p_s = at<float>(ws, L.b_ps);
  a.q_s = at<float>(ws, L.b_qs);
  a.hg_s = at<uint16_t>(ws, L.b_hgs);
  a.dp_s = at<uint16_t>(ws, L.b_dps);
  a.dq_s = at<uint16_t>(ws, L.b_dqs);
  a.dxs = at<uint16_t>(ws, L.b_dxs);
  a.dx = dx;
  a.dgate = dgate;
  a.dw1 = dw1;
  a.dw3 = dw3;
  a.dw2 = dw2;
  a.dws1 = dws1;
  a.dws3 = dws3;
  a.dws2 = dws2;
  a.accumulate = accumulate ? 1 : 0;
  a.status = st;
  a.wait_limit_ns = g_wait_limit_ns;
  a.events = g_prof_events;
  return static_cast<moe_status_t>(moe::launch_expert_backward(a, s));
}

moe_status_t moe_route_backward(const moe_dims_t* d, const float* logits,
                                const int32_t* topk_idx, const float* dgate,
                                int accumulate, float* dlogits, void* ws,
                                size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_dims(d, false));
  MOE_NEED_T(logits);
  MOE_NEED_T(topk_idx);
  MOE_NEED_T(dgate);
  MOE_NEED_T(dlogits);
  MOE_ALIGN(logits);
  MOE_ALIGN(topk_idx);
  MOE_ALIGN(dgate);
  MOE_ALIGN(dlogits);
  MOE_TRY(check_ws(d, MOE_WS_ROUTE, ws, ws_bytes));
  if (d->T == 0) return MOE_OK;
  return cuda_ok(moe::launch_route_backward(
      logits, topk_idx, dgate, d->T, d->E, d->topk, accumulate, dlogits,
      at<DevStatus>(ws, 0), cs(stream)));
}

moe_status_t moe_seq_balance_loss_backward(const moe_dims_t* d,
                                           const float* logits,
                                           int32_t seq_len, float alpha,
                                           const int32_t* counts_seq,
                                           const float* dloss, int accumulate,
                                           float* dlogits,
                                           moe_stream_t stream) {
  MOE_TRY(check_dims(d, false));
  if (seq_len < 1 || !std::isfinite(alpha)) return MOE_ERR_INVALID_ARG;
  MOE_NEED_T(logits);
  MOE_NEED_T(counts_seq);
  MOE_NEED_T(dlogits);
  MOE_ALIGN(logits);
  MOE_ALIGN(counts_seq);
  MOE_ALIGN(dloss);
  MOE_ALIGN(dlogits);
  if (d->T == 0) return MOE_OK;
  return cuda_ok(moe::launch_seq_balance_backward(
      logits, d->T, d->E, d->topk, seq_len, alpha, counts_seq, dloss,
      accumulate, dlogits, cs(stream)));
}

moe_status_t moe_route_balance_backward(
    const moe_dims_t* d, const float* logits, const int32_t* topk_idx,
    const float* dgate, int32_t seq_len, float alpha,
    const int32_t* counts_seq, const float* dloss, int accumulate,
    float* dlogits, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_dims(d, false));
  if (seq_len < 1 || !std::isfinite(alpha)) return MOE_ERR_INVALID_ARG;
  MOE_NEED_T(logits);
  MOE_NEED_T(topk_idx);
  MOE_NEED_T(dgate);
  MOE_NEED_T(counts_seq);
  MOE_NEED_T(dlogits);
  MOE_ALIGN(logits);
  MOE_ALIGN(topk_idx);
  MOE_ALIGN(dgate);
  MOE_ALIGN(counts_seq);
  MOE_ALIGN(dloss);
  MOE_ALIGN(dlogits);
  MOE_TRY(check_ws(d, MOE_WS_ROUTE, ws, ws_bytes));
  if (d->T == 0) return MOE_OK;
  return cuda_ok(moe::launch_route_balance_backward(
      logits, topk_idx, dgate, d->T, d->E, d->topk, seq_len, alpha,
      counts_seq, dloss, accumulate, dlogits, at<DevStatus>(ws, 0),
      cs(stream)));
}

moe_status_t moe_bias_update(const moe_dims_t* d, const int32_t* counts,
                             float* bias, float* load_stats,
                             moe_stream_t stream) {
  MOE_TRY(check_dims(d, false));
  MOE_NEED(counts);
  MOE_NEED(bias);
  MOE_ALIGN(counts);
  MOE_ALIGN(bias);
  MOE_ALIGN(load_stats);
  return cuda_ok(moe::launch_bias_update(counts, bias, load_stats, d->T, d->E,
                                         d->topk, d->gamma, cs(stream)));
}

moe_status_t moe_forward(const moe_dims_t* d, const moe_weights_t* w,
                         const uint16_t* x, float* bias, int update_bias,
                         uint16_t* out, float* logits_out,
                         int32_t* topk_idx_out, float* topk_gate_out,
                         int32_t* counts_out, float* load_stats_out, void* ws,
                         size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(check_dims(d, true));
  MOE_TRY(check_weights(w));
  MOE_NEED_T(x);
  MOE_NEED(bias);
  MOE_NEED_T(out);
  MOE_ALIGN(x);
  MOE_ALIGN(bias);
  MOE_ALIGN(out);
  MOE_ALIGN(logits_out);
  MOE_ALIGN(topk_idx_out);
  MOE_ALIGN(topk_gate_out);
  MOE_ALIGN(counts_out);
  MOE_ALIGN(load_stats_out);
  MOE_TRY(check_ws(d, MOE_WS_FORWARD, ws, ws_bytes));
  cudaStream_t s = cs(stream);
  const Layout L = layout(d, MOE_WS_FORWARD);
  const int T = d->T, E = d->E, K = d->topk, H = d->H;
  if (T == 0) {
    if (counts_out)
      MOE_TRY(cuda_ok(cudaMemsetAsync(counts_out, 0, sizeof(int32_t) * E, s)));
    if (update_bias || load_stats_out) {
      int32_t* cz = at<int32_t>(ws, L.counts);
      MOE_TRY(cuda_ok(cudaMemsetAsync(cz, 0, sizeof(int32_t) * E, s)));
      MOE_TRY(cuda_ok(moe::launch_bias_update(
          cz, update_bias ? bias : nullptr, load_stats_out, T, E, K, d->gamma,
          s)));
    }
    return MOE_OK;
  }
  DevStatus* st = at<DevStatus>(ws, 0);
  float* logits = logits_out ? logits_out : at<float>(ws, L.logits);
  int32_t* idx = topk_idx_out ? topk_idx_out : at<int32_t>(ws, L.idx);
  float* gate = topk_gate_out ? topk_gate_out : at<float>(ws, L.gate);
  int32_t* counts = counts_out ? counts_out : at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* dest = at<int32_t>(ws, L.dest);
  int32_t* src_row = at<int32_t>(ws, L.src_row);
  int32_t* bc = at<int32_t>(ws, L.block_counts);
  int32_t* bb = at<int32_t>(ws, L.block_base);
  uint16_t* yp = at<uint16_t>(ws, L.yp);
  uint16_t* ys = at<uint16_t>(ws, L.ys);

  prof_mark(0, s);
  MOE_TRY(router_logits_launch(
      d, x, w->w_router, w->router_offset, logits,
      at<uint16_t>(ws, L.w_split),
      L.r_partial ? at<float>(ws, L.r_partial) : nullptr, st, s,
      w->router_split));
  prof_mark(1, s);
  MOE_TRY(cuda_ok(moe::launch_route(logits, bias, T, E, d->n_group,
                                    d->topk_group, K, idx, gate, bc, s)));
  prof_mark(2, s);
  // counts, per-block prefixes -- and the bias step on this batch's load,
  // after routing consumed the old bias (same stream, so ordered)
  MOE_TRY(cuda_ok(moe::launch_scan(bc, T, E, K, counts, bb,
                                   update_bias ? bias : nullptr, d->gamma,
                                   s)));
  prof_mark(3, s);
  MOE_TRY(cuda_ok(moe::launch_dest(idx, counts, bb, T, E, K, offsets, dest,
                                   src_row, load_stats_out, st, s)));
  prof_mark(4, s);
  // few rows per expert: the up GEMM gathers them from x; else one copy
  const bool gat = gather_rows(d);
  uint16_t* xp = gat ? nullptr : at<uint16_t>(ws, L.xp);
  if (!gat) MOE_TRY(cuda_ok(moe::launch_gather(x, dest, T, H, K, xp, s)));
  prof_mark(5, s);  // 6 is recorded between the two expert GEMMs
  MOE_TRY(ffn_launch(d, w, xp, x, offsets, at<uint16_t>(ws, L.h),
                     at<uint16_t>(ws, L.hs), yp, ys, st, s,
                     g_prof_events ? g_prof_events[6] : nullptr, src_row));
  prof_mark(7, s);
  MOE_TRY(cuda_ok(moe::launch_combine(x, ys, yp, dest, gate, T, H, K, out, s)));
  prof_mark(8, s);
  return MOE_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Routing without a caller workspace.
//
// Some callers cannot hand this library any device memory beyond their
// inputs and outputs: a plugin inside a host framework that owns every
// device allocation and offers its plugins no scratch, or a latency-critical
// loop that must not call cudaMalloc after start-up (it synchronises the
// device).  For them, moe_route_static_scratch keeps the one piece of
// scratch routing needs -- the per-block expert histogram -- in the file-scope
// array below, which the CUDA runtime places on every device that loads this
// library and keeps there until the process exits.
// ---------------------------------------------------------------------------
namespace {

// The documented limit is ceil(T/64) * E <= 262144; the routing blocks of
// a batch are that count rounded up to a multiple of 148 (at most 147 more
// rows of up to 1024 experts), which the array covers.
constexpr size_t kRouteLimitInts = 262144;
constexpr size_t kRouteScratchInts = kRouteLimitInts + 147 * 1024;
static __device__ __align__(256) int32_t g_route_scratch[kRouteScratchInts];

// The address is cached per CUDA context, keyed by the context's unique id
// (cuCtxGetId, through the runtime's driver entry point so libmoe needs no
// -lcuda): after cudaDeviceReset the module may load at another address in
// the new primary context, and a cache keyed by device ordinal would hand
// the kernel a stale pointer.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct ScratchEntry {
  unsigned long long ctx_id;
  int32_t* ptr;
};
constexpr int kMaxScratchContexts = 64;
ScratchEntry g_route_scratch_ptr[kMaxScratchContexts] = {};
int g_route_scratch_n = 0;
std::mutex g_route_scratch_mu;

template <typename F>
F driver_fn(const char* name) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(f);
}

// Device address of g_route_scratch in the current context (the host-side
// name is only a stand-in for it), looked up once per context.
moe_status_t route_scratch_current_context(int32_t** out) {
  static const CtxGetCurrentFn get_ctx =
      driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (get_ctx == nullptr || get_id == nullptr) return MOE_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  if (ctx == nullptr) {
    // no context bound to this thread yet: cudaSetDevice makes the current
    // device's primary context current (it allocates nothing)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess ||
        get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr)
      return MOE_ERR_CUDA;
  }
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_route_scratch_mu);
  for (int i = 0; i < g_route_scratch_n; ++i) {
    if (g_route_scratch_ptr[i].ctx_id == id) {
      *out = g_route_scratch_ptr[i].ptr;
      return MOE_OK;
    }
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
    return MOE_ERR_CUDA;
  // a full table (more than 64 contexts over the process's life) reuses
  // the entry the id hashes to; ids are never reused, so no lookup can
  // return another context's address
  const int slot = g_route_scratch_n < kMaxScratchContexts
                       ? g_route_scratch_n++
                       : static_cast<int>(id % kMaxScratchContexts);
  g_route_scratch_ptr[slot] = {id, static_cast<int32_t*>(p)};
  *out = static_cast<int32_t*>(p);
  return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_route_static_scratch(
    const moe_dims_t* d, const float* logits, const float* bias,
    int32_t* topk_idx, float* topk_gate, int32_t* counts,
    moe_stream_t stream) {
  MOE_TRY(check_dims(d, false));
  MOE_NEED_T(logits);
  MOE_NEED(bias);
  MOE_NEED_T(topk_idx);
  MOE_NEED_T(topk_gate);
  MOE_NEED(counts);
  MOE_ALIGN(logits);
  MOE_ALIGN(bias);
  MOE_ALIGN(topk_idx);
  MOE_ALIGN(topk_gate);
  MOE_ALIGN(counts);
  // the histogram needs one row of E counts per routing block
  const size_t blocks64 =
      ((size_t)d->T + moe::kRouteTokensPerBlock - 1) /
      moe::kRouteTokensPerBlock;
  if (blocks64 * (size_t)d->E > kRouteLimitInts ||
      (size_t)moe::route_blocks(d->T) * (size_t)d->E > kRouteScratchInts)
    return MOE_ERR_WORKSPACE;
  cudaStream_t s = cs(stream);
  if (d->T == 0)
    return cuda_ok(cudaMemsetAsync(counts, 0, sizeof(int32_t) * d->E, s));
  int32_t* scratch = nullptr;
  MOE_TRY(route_scratch_current_context(&scratch));
  // every block writes its whole histogram row before the scan reads it,
  // so nothing left from an earlier call needs clearing
  MOE_TRY(cuda_ok(moe::launch_route(logits, bias, d->T, d->E, d->n_group,
                                    d->topk_group, d->topk, topk_idx,
                                    topk_gate, scratch, s)));
  return cuda_ok(moe::launch_scan(scratch, d->T, d->E, d->topk, counts,
                                  nullptr, nullptr, 0.f, s));
}
