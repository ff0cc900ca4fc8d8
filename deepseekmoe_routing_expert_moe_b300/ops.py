"""ctypes binding of libmoe.so -- argument marshalling only.

Each function has the name of the C entry point it calls (include/moe.h)
and takes torch CUDA tensors; torch provides device memory and the current
stream, nothing else.  Every step of the layer runs in the library's CUDA
kernels.  There is no fallback: if the library is missing or a call fails,
an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe.so")

(MOE_WS_ROUTE, MOE_WS_PERMUTE, MOE_WS_EXPERT_FFN, MOE_WS_FORWARD,
 MOE_WS_ROUTER_LOGITS, MOE_WS_SEQ_BALANCE, MOE_WS_EXPERT_FFN_FP8,
 MOE_WS_EXPERT_BWD, MOE_WS_EXPERT_FFN_MX) = 0, 1, 2, 3, 4, 5, 6, 7, 8

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_ALIGNMENT", 4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA",
          6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_DEVICE_BOUNDS"}
STATUS_CODES = {v: k for k, v in STATUS.items()}


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


class MoeDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32),
                ("E", ctypes.c_int32), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("I", ctypes.c_int32), ("I_shared", ctypes.c_int32),
                ("gamma", ctypes.c_float)]


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_router", "w1", "w3", "w2", "ws1", "ws3", "ws2",
                 "router_offset", "router_split")]


class MoeWeightsFp8(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w1", "w1_scale", "w3", "w3_scale", "w2", "w2_scale",
                 "ws1", "ws1_scale", "ws3", "ws3_scale", "ws2", "ws2_scale")]


class MoeWeightsMx(MoeWeightsFp8):
    """moe_weights_mx_t: the same twelve pointers (UE8M0 byte scales)."""


_P = ctypes.c_void_p
_D = ctypes.POINTER(MoeDims)
_W = ctypes.POINTER(MoeWeights)
_S = ctypes.c_size_t
_I = ctypes.c_int
_SIGS = {
    "moe_workspace_bytes": (ctypes.c_size_t, [_D, _I]),
    "moe_router_logits": (_I, [_D, _P, _P, _P, _P, _P, _S, _P]),
    "moe_route": (_I, [_D, _P, _P, _P, _P, _P, _P, _S, _P]),
    "moe_route_static_scratch": (_I, [_D, _P, _P, _P, _P, _P, _P]),
    "moe_permute": (_I, [_D, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "moe_expert_ffn": (_I, [_D, _W, _P, _P, _P, _P, _P, _P, _S, _P]),
    "moe_combine": (_I, [_D, _P, _P, _P, _P, _P, _P, _P]),
    "moe_expert_ffn_routed": (_I, [_D, _W, _P, _P, _P, _P, _S, _P]),
    "moe_ep_plan": (_I, [ctypes.c_int32, ctypes.c_int32, _P, ctypes.c_int64,
                         _P, _P, _P, _P]),
    "moe_ep_permute_rows": (_I, [_P, ctypes.c_int64, ctypes.c_int64, _P,
                                 ctypes.c_int32, _P, _P, _P]),
    "moe_bias_update": (_I, [_D, _P, _P, _P, _P]),
    "moe_seq_balance_loss": (_I, [_D, _P, ctypes.c_int32, ctypes.c_float, _P,
                                  _P, _P, _P, _S, _P]),
    "moe_quantize_fp8_blocks": (_I, [_P, ctypes.c_int64, ctypes.c_int64, _P,
                                     _P, _P]),
    "moe_quantize_fp8_rows": (_I, [_P, ctypes.c_int64, ctypes.c_int64, _P,
                                   _P, _P]),
    "moe_permute_fp8": (_I, [_D, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "moe_expert_ffn_fp8": (_I, [_D, ctypes.POINTER(MoeWeightsFp8), _P, _P,
                                _P, _P, _P, _P, _P, _P, _S, _P]),
    "moe_quantize_mx_blocks": (_I, [_P, ctypes.c_int64, ctypes.c_int64, _P,
                                    _P, _P]),
    "moe_quantize_mx_rows": (_I, [_P, ctypes.c_int64, ctypes.c_int64, _P,
                                  _P, _P]),
    "moe_permute_mx": (_I, [_D, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "moe_expert_ffn_mx": (_I, [_D, ctypes.POINTER(MoeWeightsMx), _P, _P,
                               _P, _P, _P, _P, _P, _P, _S, _P]),
    "moe_expert_ffn_mx_routed": (_I, [_D, ctypes.POINTER(MoeWeightsMx), _P,
                                      _P, _P, _P, _P, _S, _P]),
    "moe_plan_redundant_experts": (_I, [_P, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int32, _P, _P]),
    "moe_route_backward": (_I, [_D, _P, _P, _P, _I, _P, _P, _S, _P]),
    "moe_expert_backward": (_I, [_D, _W, _P, _P, _P, _P, _I, _P, _P, _P, _P,
                                 _P, _P, _P, _P, _P, _S, _P]),
    "moe_seq_balance_loss_backward": (_I, [_D, _P, ctypes.c_int32,
                                           ctypes.c_float, _P, _P, _I, _P,
                                           _P]),
    "moe_route_balance_backward": (_I, [_D, _P, _P, _P, ctypes.c_int32,
                                        ctypes.c_float, _P, _P, _I, _P, _P,
                                        _S, _P]),
    "moe_forward": (_I, [_D, _W, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _S,
                         _P]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_get_device_error": (_I, [_P, _P]),
    "moe_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "moe_set_gemm_ctas": (None, [ctypes.c_int32]),
    "moe_abi_version": (ctypes.c_int32, []),
    "moe_router_weight_split": (_I, [_P, ctypes.c_int32, ctypes.c_int32,
                                     _P, _P]),
    "moe_set_profile_events": (None, [ctypes.POINTER(ctypes.c_void_p),
                                       ctypes.c_int32]),
}

MOE_FORWARD_KERNELS = 8
FORWARD_KERNEL_NAMES = ("router_logits", "route", "scan", "dest", "gather",
                        "gemm_up_swiglu", "gemm_down", "combine")

_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing; build it with "
                "`python -m deepseekmoe_routing_expert_moe_b300.build` "
                "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


# ------------------------------------------------------------ marshalling
def dims(T, H, E, n_group, topk_group, topk, I=64, I_shared=64,
         gamma=0.001) -> MoeDims:
    return MoeDims(T, H, E, n_group, topk_group, topk, I, I_shared, gamma)


def dims_of(cfg, **over) -> MoeDims:
    return dims(**cfg.dims(**over))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(fn: str, code: int):
    if code != 0:
        raise MoeError(fn, code)


class Weights:
    """Device weights of one layer (torch tensors; bf16 stored as int16)."""

    def __init__(self, w_router, w1, w3, w2, ws1, ws3, ws2,
                 router_offset=None, router_split=None):
        self.w_router, self.w1, self.w3, self.w2 = w_router, w1, w3, w2
        self.ws1, self.ws3, self.ws2 = ws1, ws3, ws2
        self.router_offset = router_offset
        self.router_split = router_split
        self.struct = MoeWeights(*(_ptr(t) for t in (w_router, w1, w3, w2,
                                                      ws1, ws3, ws2,
                                                      router_offset,
                                                      router_split)))

    def with_router_split(self, stream=None):
        """The same weights with the router weight's bf16 split made once
        (moe_router_weight_split), so moe_forward does not redo it."""
        E, H = self.w_router.shape
        split = torch.empty((3, E, H), dtype=torch.int16,
                            device=self.w_router.device)
        moe_router_weight_split(self.w_router, split, stream)
        return Weights(self.w_router, self.w1, self.w3, self.w2, self.ws1,
                       self.ws3, self.ws2, self.router_offset, split)


class WeightsFp8:
    """FP8 expert weights: (codes uint8, block scales fp32) pairs for w1,
    w3, w2 (all experts) and ws1, ws3, ws2 (shared expert)."""

    NAMES = ("w1", "w3", "w2", "ws1", "ws3", "ws2")

    def __init__(self, **pairs):
        self.pairs = pairs
        flat = []
        for n in self.NAMES:
            q, s = pairs[n]
            flat += [_ptr(q), _ptr(s)]
        self.struct = MoeWeightsFp8(*flat)

    @classmethod
    def quantize(cls, w1, w3, w2, ws1, ws3, ws2, stream=None):
        """128 x 128 block quantization of bf16 (int16) weights on the
        device: w1, w3 [E, I, H], w2 [E, H, I], ws1, ws3 [I_s, H],
        ws2 [H, I_s]."""
        pairs = {}
        for n, t in zip(cls.NAMES, (w1, w3, w2, ws1, ws3, ws2)):
            t2 = t.reshape(-1, t.shape[-1])
            q = torch.empty(t2.shape, dtype=torch.uint8, device=t.device)
            s = torch.empty((t2.shape[0] // 128, t2.shape[1] // 128),
                            dtype=torch.float32, device=t.device)
            moe_quantize_fp8_blocks(t2, q, s, stream)
            pairs[n] = (q, s)
        return cls(**pairs)


class WeightsMx(WeightsFp8):
    """FP8 expert weights with power-of-two scales: (codes uint8, UE8M0
    block scales uint8) pairs for w1, w3, w2 and ws1, ws3, ws2."""

    def __init__(self, **pairs):
        """(codes, scales) pairs by name; a name left out (the shared expert
        of moe_expert_ffn_mx_routed's weights) is passed as NULL."""
        self.pairs = pairs
        flat = []
        for n in self.NAMES:
            q, s = pairs.get(n, (None, None))
            flat += [_ptr(q), _ptr(s)]
        self.struct = MoeWeightsMx(*flat)

    @classmethod
    def quantize(cls, w1, w3, w2, ws1, ws3, ws2, stream=None):
        """128 x 128 block quantization with power-of-two scales of bf16
        (int16) weights on the device (shapes as WeightsFp8.quantize)."""
        pairs = {}
        for n, t in zip(cls.NAMES, (w1, w3, w2, ws1, ws3, ws2)):
            t2 = t.reshape(-1, t.shape[-1])
            q = torch.empty(t2.shape, dtype=torch.uint8, device=t.device)
            s = torch.empty((t2.shape[0] // 128, t2.shape[1] // 128),
                            dtype=torch.uint8, device=t.device)
            moe_quantize_mx_blocks(t2, q, s, stream)
            pairs[n] = (q, s)
        return cls(**pairs)


def workspace_bytes(d: MoeDims, which: int) -> int:
    return lib().moe_workspace_bytes(ctypes.byref(d), which)


def workspace(d: MoeDims, which: int, device="cuda") -> torch.Tensor:
    """A zeroed device workspace sized for entry point `which`."""
    n = workspace_bytes(d, which)
    if n == 0:
        raise MoeError("moe_workspace_bytes", 1)
    return torch.zeros(n, dtype=torch.uint8, device=device)


# ----------------------------------------------------------- entry points
def moe_router_logits(d, x, w_router, logits, ws, router_offset=None,
                      stream=None):
    _check("moe_router_logits", lib().moe_router_logits(
        ctypes.byref(d), _ptr(x), _ptr(w_router), _ptr(router_offset),
        _ptr(logits), _ptr(ws), ws.numel(), _stream(stream)))


def moe_route(d, logits, bias, topk_idx, topk_gate, counts, ws, stream=None):
    _check("moe_route", lib().moe_route(
        ctypes.byref(d), _ptr(logits), _ptr(bias), _ptr(topk_idx),
        _ptr(topk_gate), _ptr(counts), _ptr(ws), ws.numel(), _stream(stream)))


def moe_route_static_scratch(d, logits, bias, topk_idx, topk_gate, counts,
                             stream=None):
    """moe_route without a workspace (its scratch is a static device array;
    concurrent calls on overlapping streams race on it)."""
    _check("moe_route_static_scratch", lib().moe_route_static_scratch(
        ctypes.byref(d), _ptr(logits), _ptr(bias), _ptr(topk_idx),
        _ptr(topk_gate), _ptr(counts), _stream(stream)))


def moe_permute(d, x, topk_idx, offsets, dest, src_row, xp, ws, stream=None):
    _check("moe_permute", lib().moe_permute(
        ctypes.byref(d), _ptr(x), _ptr(topk_idx), _ptr(offsets), _ptr(dest),
        _ptr(src_row), _ptr(xp), _ptr(ws), ws.numel(), _stream(stream)))


def moe_expert_ffn(d, w: Weights, xp, x, offsets, yp, ys, ws, stream=None):
    _check("moe_expert_ffn", lib().moe_expert_ffn(
        ctypes.byref(d), ctypes.byref(w.struct), _ptr(xp), _ptr(x),
        _ptr(offsets), _ptr(yp), _ptr(ys), _ptr(ws), ws.numel(),
        _stream(stream)))


def moe_expert_ffn_routed(d, w: Weights, xp, offsets, yp, ws, stream=None):
    """Routed experts only over d.T * d.topk expert-sorted rows."""
    _check("moe_expert_ffn_routed", lib().moe_expert_ffn_routed(
        ctypes.byref(d), ctypes.byref(w.struct), _ptr(xp), _ptr(offsets),
        _ptr(yp), _ptr(ws), ws.numel(), _stream(stream)))


def moe_ep_plan(counts, rows, perm, offsets_local, ws=None, stream=None):
    """counts: [n_src, n_local] int32 device tensor."""
    n_src, n_local = counts.shape
    _check("moe_ep_plan", lib().moe_ep_plan(
        n_src, n_local, _ptr(counts), int(rows), _ptr(perm),
        _ptr(offsets_local), _ptr(ws), _stream(stream)))


def moe_ep_permute_rows(inp, perm, out, inverse=False, ws=None, stream=None):
    """Rows of a 2-D device tensor moved by an expert-parallel map."""
    rows = inp.shape[0]
    row_bytes = inp.numel() * inp.element_size() // max(rows, 1)
    _check("moe_ep_permute_rows", lib().moe_ep_permute_rows(
        _ptr(inp), rows, row_bytes, _ptr(perm), 1 if inverse else 0,
        _ptr(out), _ptr(ws), _stream(stream)))


def moe_combine(d, x, ys, yp, dest, topk_gate, out, stream=None):
    _check("moe_combine", lib().moe_combine(
        ctypes.byref(d), _ptr(x), _ptr(ys), _ptr(yp), _ptr(dest),
        _ptr(topk_gate), _ptr(out), _stream(stream)))


def moe_bias_update(d, counts, bias, load_stats=None, stream=None):
    _check("moe_bias_update", lib().moe_bias_update(
        ctypes.byref(d), _ptr(counts), _ptr(bias), _ptr(load_stats),
        _stream(stream)))


def moe_seq_balance_loss(d, logits, seq_len, alpha, counts_seq, P_seq, loss,
                         ws, stream=None):
    """Per-sequence balance loss: counts_seq [n_seq, E] int32, P_seq
    [n_seq, E] fp32, loss [n_seq] fp32, n_seq = ceil(T / seq_len)."""
    _check("moe_seq_balance_loss", lib().moe_seq_balance_loss(
        ctypes.byref(d), _ptr(logits), int(seq_len), float(alpha),
        _ptr(counts_seq), _ptr(P_seq), _ptr(loss), _ptr(ws), ws.numel(),
        _stream(stream)))


def moe_quantize_fp8_blocks(w, q, scale, stream=None):
    """128 x 128 block E4M3 quantization of a 2-D bf16 (int16) tensor."""
    rows, cols = w.shape
    _check("moe_quantize_fp8_blocks", lib().moe_quantize_fp8_blocks(
        _ptr(w), rows, cols, _ptr(q), _ptr(scale), _stream(stream)))


def moe_quantize_fp8_rows(x, q, scale, stream=None):
    """1 x 128 tile E4M3 quantization of a 2-D bf16 (int16) tensor."""
    rows, cols = x.shape
    _check("moe_quantize_fp8_rows", lib().moe_quantize_fp8_rows(
        _ptr(x), rows, cols, _ptr(q), _ptr(scale), _stream(stream)))


def moe_permute_fp8(d, x, dest, xq, xs, xpq, xps, ws, stream=None):
    _check("moe_permute_fp8", lib().moe_permute_fp8(
        ctypes.byref(d), _ptr(x), _ptr(dest), _ptr(xq), _ptr(xs), _ptr(xpq),
        _ptr(xps), _ptr(ws), ws.numel(), _stream(stream)))


def moe_expert_ffn_fp8(d, w: WeightsFp8, xpq, xps, xq, xs, offsets, yp, ys,
                       ws, stream=None):
    _check("moe_expert_ffn_fp8", lib().moe_expert_ffn_fp8(
        ctypes.byref(d), ctypes.byref(w.struct), _ptr(xpq), _ptr(xps),
        _ptr(xq), _ptr(xs), _ptr(offsets), _ptr(yp), _ptr(ys), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_quantize_mx_blocks(w, q, scale, stream=None):
    """128 x 128 block E4M3 quantization with power-of-two (UE8M0) scales of
    a 2-D bf16 (int16) tensor."""
    rows, cols = w.shape
    _check("moe_quantize_mx_blocks", lib().moe_quantize_mx_blocks(
        _ptr(w), rows, cols, _ptr(q), _ptr(scale), _stream(stream)))


def moe_quantize_mx_rows(x, q, scale, stream=None):
    """1 x 128 tile E4M3 quantization with power-of-two (UE8M0) scales of a
    2-D bf16 (int16) tensor."""
    rows, cols = x.shape
    _check("moe_quantize_mx_rows", lib().moe_quantize_mx_rows(
        _ptr(x), rows, cols, _ptr(q), _ptr(scale), _stream(stream)))


def moe_permute_mx(d, x, dest, xq, xs, xpq, xps, ws, stream=None):
    _check("moe_permute_mx", lib().moe_permute_mx(
        ctypes.byref(d), _ptr(x), _ptr(dest), _ptr(xq), _ptr(xs), _ptr(xpq),
        _ptr(xps), _ptr(ws), ws.numel(), _stream(stream)))


def moe_expert_ffn_mx(d, w: WeightsMx, xpq, xps, xq, xs, offsets, yp, ys,
                      ws, stream=None):
    _check("moe_expert_ffn_mx", lib().moe_expert_ffn_mx(
        ctypes.byref(d), ctypes.byref(w.struct), _ptr(xpq), _ptr(xps),
        _ptr(xq), _ptr(xs), _ptr(offsets), _ptr(yp), _ptr(ys), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_expert_ffn_mx_routed(d, w: WeightsMx, xpq, xps, offsets, yp, ws,
                             stream=None):
    _check("moe_expert_ffn_mx_routed", lib().moe_expert_ffn_mx_routed(
        ctypes.byref(d), ctypes.byref(w.struct), _ptr(xpq), _ptr(xps),
        _ptr(offsets), _ptr(yp), _ptr(ws), ws.numel(), _stream(stream)))


def moe_plan_redundant_experts(load, n_devices, slots_per_device):
    """Host planner: load [E] (numpy int64) -> (slot_expert [D, r] int32,
    device_load [D] int64)."""
    import numpy as np
    load = np.ascontiguousarray(load, np.int64)
    D, r = int(n_devices), int(slots_per_device)
    slots = np.full((D, r), -7, np.int32)
    dl = np.zeros(D, np.int64)
    _check("moe_plan_redundant_experts", lib().moe_plan_redundant_experts(
        load.ctypes.data, load.shape[0], D, r,
        slots.ctypes.data if D * r else None, dl.ctypes.data))
    return slots, dl


def moe_route_backward(d, logits, topk_idx, dgate, dlogits, ws,
                       accumulate=False, stream=None):
    _check("moe_route_backward", lib().moe_route_backward(
        ctypes.byref(d), _ptr(logits), _ptr(topk_idx), _ptr(dgate),
        1 if accumulate else 0, _ptr(dlogits), _ptr(ws), ws.numel(),
        _stream(stream)))


class WeightGrads:
    """fp32 weight gradients of one layer's experts: dw1, dw3 [E, I, H],
    dw2 [E, H, I], dws1, dws3 [I_s, H], dws2 [H, I_s] (torch tensors)."""

    NAMES = ("dw1", "dw3", "dw2", "dws1", "dws3", "dws2")

    def __init__(self, dw1, dw3, dw2, dws1, dws3, dws2):
        self.dw1, self.dw3, self.dw2 = dw1, dw3, dw2
        self.dws1, self.dws3, self.dws2 = dws1, dws3, dws2

    @classmethod
    def empty(cls, d, device="cuda"):
        E, H, I, Is = d.E, d.H, d.I, d.I_shared
        f = lambda *s: torch.empty(s, dtype=torch.float32, device=device)  # noqa: E731
        return cls(f(E, I, H), f(E, I, H), f(E, H, I), f(Is, H), f(Is, H),
                   f(H, Is))

    def tensors(self):
        return [getattr(self, n) for n in self.NAMES]


def moe_expert_backward(d, w: Weights, x, dout, topk_idx, topk_gate, dx,
                        dgate, grads: WeightGrads, ws, accumulate=False,
                        stream=None):
    _check("moe_expert_backward", lib().moe_expert_backward(
        ctypes.byref(d), ctypes.byref(w.struct), _ptr(x), _ptr(dout),
        _ptr(topk_idx), _ptr(topk_gate), 1 if accumulate else 0, _ptr(dx),
        _ptr(dgate), *(_ptr(t) for t in grads.tensors()), _ptr(ws),
        ws.numel(), _stream(stream)))


def moe_seq_balance_loss_backward(d, logits, seq_len, alpha, counts_seq,
                                  dlogits, dloss=None, accumulate=False,
                                  stream=None):
    _check("moe_seq_balance_loss_backward",
           lib().moe_seq_balance_loss_backward(
               ctypes.byref(d), _ptr(logits), int(seq_len), float(alpha),
               _ptr(counts_seq), _ptr(dloss), 1 if accumulate else 0,
               _ptr(dlogits), _stream(stream)))


def moe_route_balance_backward(d, logits, topk_idx, dgate, seq_len, alpha,
                               counts_seq, dlogits, ws, dloss=None,
                               accumulate=False, stream=None):
    _check("moe_route_balance_backward",
           lib().moe_route_balance_backward(
               ctypes.byref(d), _ptr(logits), _ptr(topk_idx), _ptr(dgate),
               int(seq_len), float(alpha), _ptr(counts_seq), _ptr(dloss),
               1 if accumulate else 0, _ptr(dlogits), _ptr(ws), ws.numel(),
               _stream(stream)))


def moe_forward(d, w: Weights, x, bias, out, ws, update_bias=False,
                logits_out=None, topk_idx_out=None, topk_gate_out=None,
                counts_out=None, load_stats_out=None, stream=None):
    _check("moe_forward", lib().moe_forward(
        ctypes.byref(d), ctypes.byref(w.struct), _ptr(x), _ptr(bias),
        1 if update_bias else 0, _ptr(out), _ptr(logits_out),
        _ptr(topk_idx_out), _ptr(topk_gate_out), _ptr(counts_out),
        _ptr(load_stats_out), _ptr(ws), ws.numel(), _stream(stream)))


def moe_get_device_error(ws, stream=None) -> int:
    return lib().moe_get_device_error(_ptr(ws), _stream(stream))


def moe_set_wait_timeout_ns(ns: int):
    lib().moe_set_wait_timeout_ns(ns)


def moe_set_gemm_ctas(n: int):
    """Cap the expert GEMMs' persistent grid at n CTAs (0 = one per SM)."""
    lib().moe_set_gemm_ctas(n)


_prof_keep = None


def moe_set_profile_events(events):
    """events: a list of MOE_FORWARD_KERNELS + 1 torch.cuda.Event (enabled
    for timing), or None to disable."""
    global _prof_keep
    if events is None:
        _prof_keep = None
        lib().moe_set_profile_events(None, 0)
        return
    for e in events:        # torch creates the CUDA event on first record
        e.record()
    torch.cuda.synchronize()
    arr = (ctypes.c_void_p * len(events))(*(e.cuda_event for e in events))
    _prof_keep = (events, arr)
    lib().moe_set_profile_events(arr, len(events))


def moe_status_string(code: int) -> str:
    return lib().moe_status_string(code).decode()


def moe_router_weight_split(w_router, split, stream=None):
    """w_router [E, H] fp32 -> split [3, E, H] bf16 (as int16)."""
    E, H = w_router.shape
    _check("moe_router_weight_split", lib().moe_router_weight_split(
        _ptr(w_router), E, H, _ptr(split), _stream(stream)))


def moe_abi_version() -> int:
    return lib().moe_abi_version()
