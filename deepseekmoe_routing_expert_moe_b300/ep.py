"""Expert-parallel layer forward across ranks ("02 · DeepSeek-V3" §1.3
node-limited routing, §2 dispatch / combine, §5.1 EP deployment).

Rank r of P holds the routed experts [r*El, (r+1)*El) (El = E / P) and a
replica of the router and the shared expert.  Per step, on every rank:

  1. route its own tokens (router logits, sigmoid + bias, group-limited
     top-K, gates, load histogram);
  2. dispatch: the expert-sorted rows of the stable permutation are already
     grouped by destination rank, so the send buffer is that permutation;
     the per-(destination, expert) counts are exchanged first, then the rows
     (one all-to-all each);
  3. regroup the received rows from source-major to expert-major order and
     run the rank's experts as one grouped GEMM (routed rows only);
  4. send the outputs back (the inverse regroup, one all-to-all) and combine
     them with the gates, the shared expert and the residual;
  5. bias step on the global load (an all-reduce of the count vector).

With n_group = P (a group per rank, the pages' node-limited routing) every
token's rows go to at most topk_group ranks.

The arithmetic runs in a backend; ``CudaBackend`` calls this library's C
ABI (there is no fallback: it raises when the library is missing).  The
exchanges use ``torch.distributed``: NCCL exchanges device tensors; with a
gloo group the rows are staged through host memory.

Dispatch in FP8 (same page, §2: activations are cast to FP8 before they are
sent, the outputs return in BF16): with ``CudaBackend(..., mx=...)`` a rank
quantizes its tokens once (E4M3 codes with power-of-two 1 x 128 scales,
``moe_permute_mx``), sends the expert-sorted codes and their scale bytes
(1 + 1/128 bytes per value instead of 2), the receiver runs its experts on
them (``moe_expert_ffn_mx_routed``) and returns bf16 rows; the shared
expert runs on the same codes.  A backend's ``permute`` may return the rows
as a tuple of tensors with the same leading dimension (codes, scales): each
is exchanged and regrouped alike.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist


class CudaBackend:
    """The per-rank arithmetic on this GPU through the C ABI (ops.py)."""

    def __init__(self, cfg_dims, weights, local_weights, rank, world,
                 device="cuda", mx=None):
        from . import ops
        self.ops = ops
        self.d = cfg_dims              # global layer dims (ops.MoeDims)
        self.W = weights               # ops.Weights: router, shared expert
        self.Wl = local_weights        # ops.Weights: this rank's experts
        self.rank, self.world = rank, world
        self.device = device
        # FP8 dispatch: mx = (ops.WeightsMx of this rank's experts,
        # ops.WeightsMx holding the shared expert as one expert), or None
        self.mx = mx
        self._tok_q = None             # this step's token codes and scales
        self._ws = {}

    def _workspace(self, d, which):
        key = (d.T, d.topk, d.E, d.I, which)
        if key not in self._ws:
            self._ws[key] = self.ops.workspace(d, which, self.device)
        return self._ws[key]

    def route(self, x, bias):
        o, d = self.ops, self.d
        T, E, K = d.T, d.E, d.topk
        z = torch.empty((T, E), dtype=torch.float32, device=self.device)
        ws = self._workspace(d, o.MOE_WS_ROUTER_LOGITS)
        o.moe_router_logits(d, x, self.W.w_router, z, ws,
                            router_offset=self.W.router_offset)
        idx = torch.empty((T, K), dtype=torch.int32, device=self.device)
        gate = torch.empty((T, K), dtype=torch.float32, device=self.device)
        counts = torch.empty(E, dtype=torch.int32, device=self.device)
        o.moe_route(d, z, bias, idx, gate, counts,
                    self._workspace(d, o.MOE_WS_ROUTE))
        return idx, gate, counts

    def permute(self, x, idx):
        o, d = self.ops, self.d
        T, E, K, H = d.T, d.E, d.topk, d.H
        offsets = torch.empty(E + 1, dtype=torch.int32, device=self.device)
        dest = torch.empty((T, K), dtype=torch.int32, device=self.device)
        src = torch.empty(T * K, dtype=torch.int32, device=self.device)
        ws = self._workspace(d, o.MOE_WS_PERMUTE)
        if self.mx is None:
            xp = torch.empty((T * K, H), dtype=torch.int16,
                             device=self.device)
            o.moe_permute(d, x, idx, offsets, dest, src, xp, ws)
            return offsets, dest, xp
        # FP8 dispatch: the indices, then the tokens quantized once and
        # their codes and scales copied to the expert-sorted rows
        o.moe_permute(d, None, idx, offsets, dest, src, None, ws)
        u8 = dict(dtype=torch.uint8, device=self.device)
        xq = torch.empty((T, H), **u8)
        xs = torch.empty((T, H // 128), **u8)
        xpq = torch.empty((T * K, H), **u8)
        xps = torch.empty((T * K, H // 128), **u8)
        o.moe_permute_mx(d, x, dest, xq, xs, xpq, xps, ws)
        self._tok_q = (xq, xs)
        return offsets, dest, (xpq, xps)

    def plan(self, recv_counts, rows):
        n_local = recv_counts.shape[1]
        perm = torch.empty(max(rows, 1), dtype=torch.int32,
                           device=self.device)
        off = torch.empty(n_local + 1, dtype=torch.int32, device=self.device)
        self.ops.moe_ep_plan(recv_counts.contiguous(), rows, perm, off)
        return perm, off

    def permute_rows(self, rows, perm, inverse):
        out = torch.empty_like(rows)
        if rows.shape[0]:
            self.ops.moe_ep_permute_rows(rows, perm, out, inverse=inverse)
        return out

    def _local_dims(self, n_rows, n_experts):
        d = self.d
        return self.ops.dims(n_rows, d.H, n_experts, 1, 1, 1, d.I,
                             d.I_shared, d.gamma)

    def experts(self, xr, offsets_local):
        o = self.ops
        if self.mx is not None:
            codes, scales = xr
            R = codes.shape[0]
            yr = torch.empty((R, self.d.H), dtype=torch.int16,
                             device=self.device)
            if R:
                dl = self._local_dims(R, offsets_local.shape[0] - 1)
                o.moe_expert_ffn_mx_routed(
                    dl, self.mx[0], codes, scales, offsets_local, yr,
                    self._workspace(dl, o.MOE_WS_EXPERT_FFN_MX))
            return yr
        R = xr.shape[0]
        yr = torch.empty_like(xr)
        if R == 0:
            return yr
        dl = self._local_dims(R, offsets_local.shape[0] - 1)
        o.moe_expert_ffn_routed(dl, self.Wl, xr, offsets_local, yr,
                                self._workspace(dl, o.MOE_WS_EXPERT_FFN))
        return yr

    def shared(self, x):
        """The shared expert as a one-expert routed FFN over the tokens (on
        the step's token codes when dispatching in FP8)."""
        o, d = self.ops, self.d
        T = x.shape[0]
        ys = torch.empty_like(x)
        if T == 0:
            return ys
        dl = self._local_dims(T, 1)
        off = torch.tensor([0, T], dtype=torch.int32, device=self.device)
        if self.mx is not None:
            dl.I = d.I_shared
            xq, xs = self._tok_q
            o.moe_expert_ffn_mx_routed(
                dl, self.mx[1], xq, xs, off, ys,
                self._workspace(dl, o.MOE_WS_EXPERT_FFN_MX))
            return ys
        Ws = o.Weights(self.W.w_router, self.W.ws1.unsqueeze(0),
                       self.W.ws3.unsqueeze(0), self.W.ws2.unsqueeze(0),
                       self.W.ws1, self.W.ws3, self.W.ws2)
        dl.I = d.I_shared
        o.moe_expert_ffn_routed(dl, Ws, x, off, ys,
                                self._workspace(dl, o.MOE_WS_EXPERT_FFN))
        return ys

    def combine(self, x, ys, yp, dest, gate):
        out = torch.empty_like(x)
        self.ops.moe_combine(self.d, x, ys, yp, dest, gate, out)
        return out

    def bias_update(self, counts_global, bias, tokens_global):
        d = self.ops.dims(tokens_global, self.d.H, self.d.E, self.d.n_group,
                          self.d.topk_group, self.d.topk, self.d.I,
                          self.d.I_shared, self.d.gamma)
        self.ops.moe_bias_update(d, counts_global, bias)


def _exchange(group, out, inp, out_splits, in_splits):
    """all_to_all_single of the rows of 2-D tensors (any dtype, moved as
    bytes, so bf16 bits travel unchanged); with a gloo group the rows go
    through host memory."""
    rb = inp.element_size() * (inp.shape[1] if inp.dim() > 1 else 1)
    ob = out.view(torch.uint8).reshape(-1)
    ib = inp.view(torch.uint8).reshape(-1)
    osz = [int(s) * rb for s in out_splits]
    isz = [int(s) * rb for s in in_splits]
    if dist.get_backend(group) == "gloo" and ib.is_cuda:
        oh = torch.empty(ob.numel(), dtype=torch.uint8)
        dist.all_to_all_single(oh, ib.cpu(), osz, isz, group=group)
        ob.copy_(oh.to(ob.device))
    else:
        dist.all_to_all_single(ob, ib, osz, isz, group=group)


def _all_reduce(group, t):
    if dist.get_backend(group) == "gloo" and t.is_cuda:
        h = t.cpu()
        dist.all_reduce(h, group=group)
        t.copy_(h.to(t.device))
    else:
        dist.all_reduce(t, group=group)


class ExpertParallel:
    """One rank's side of the expert-parallel layer forward (see the module
    docstring).  ``backend`` does the arithmetic, ``group`` the exchanges."""

    def __init__(self, backend, E, topk, topk_group, n_group, group=None):
        self.be = backend
        self.group = group
        self.P = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if E % self.P:
            raise ValueError("the experts must split evenly over the ranks")
        self.E, self.El, self.K = E, E // self.P, topk
        self.topk_group, self.n_group = topk_group, n_group
        self.last = {}

    def forward(self, x, bias, update_bias=True):
        be, P, El = self.be, self.P, self.El
        T, H = x.shape
        idx, gate, counts = be.route(x, bias)
        offsets, dest, rows = be.permute(x, idx)
        parts = rows if isinstance(rows, tuple) else (rows,)
        off = np.asarray(offsets.cpu()).astype(np.int64)
        send = [int(off[(r + 1) * El] - off[r * El]) for r in range(P)]
        # counts of my experts from every source, [P, El]
        recv_counts = torch.empty_like(counts)
        _exchange(self.group, recv_counts.view(P, El), counts.view(P, El),
                  [1] * P, [1] * P)
        rc = np.asarray(recv_counts.cpu()).astype(np.int64).reshape(P, El)
        recv = [int(v) for v in rc.sum(1)]
        R = sum(recv)
        # the dispatch: every part of the rows (bf16 rows, or E4M3 codes and
        # their scale bytes), then each regrouped alike
        received = []
        for part in parts:
            dst = torch.empty((R, part.shape[1]), dtype=part.dtype,
                              device=part.device)
            _exchange(self.group, dst, part, recv, send)
            received.append(dst)
        perm, off_local = be.plan(recv_counts.view(P, El), R)
        xr = tuple(be.permute_rows(p, perm, inverse=False) for p in received)
        yr = be.experts(xr if isinstance(rows, tuple) else xr[0], off_local)
        yr_src = be.permute_rows(yr, perm, inverse=True)
        # the return trip: the experts' outputs in BF16
        yp = torch.empty((parts[0].shape[0], H), dtype=yr.dtype,
                         device=yr.device)
        _exchange(self.group, yp, yr_src, send, recv)
        ys = be.shared(x)
        out = be.combine(x, ys, yp, dest, gate)
        if update_bias:
            g = counts.clone()
            _all_reduce(self.group, g)
            be.bias_update(g, bias, T * P)
        self.last = dict(idx=idx, gate=gate, counts=counts, send=send,
                         recv=recv, recv_counts=rc)
        return out
