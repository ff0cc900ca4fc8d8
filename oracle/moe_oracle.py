"""CPU oracle for the DeepSeekMoE layer forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` legs may import this module.  It
shares no code, header, table or constant with the CUDA path and imports
nothing from the product package; the two meet only through the seeded input
generator, which holds none of the method's arithmetic.

What it computes, and where the pages say so (page titles as cited):

* "02 · DeepSeek-V3" (PaperTrace) §1.3, eq. 12/13/15: the MoE output is the
  residual plus the shared expert plus the gate-weighted sum of the routed
  experts; affinities are sigmoids of the router scores; gates are the
  chosen affinities normalised over the chosen top-8 (so they sum to 1).
* same page §1.3, node-limited routing: experts fall into groups; a group's
  score is the sum of its K_r/M = 2 highest affinities; the best 4 groups are
  kept and top-8 is taken only among their experts.
* same page §1.4, eq. 16: a per-expert bias b_i is added to the affinity for
  the top-K selection only; the gate still uses the raw affinity; at step end
  overloaded experts get b_i -= gamma and underloaded ones b_i += gamma,
  gamma = 0.001.
* same page §1.1: every expert is a SwiGLU FFN with three matrices
  (7168 x 2048 each for V3).
* same page §1.4, eq. 17-20: the sequence-wise balance loss
  alpha * sum_i f_i P_i (alpha = 1e-4), and its gradient to the logits
  together with the gates' (the routing backward).
* same page §2: FP8 (E4M3) with one scale per 1 x 128 activation tile and
  128 x 128 weight block, and the expert FFN on those values; the same
  groups with power-of-two scales (the microscaling form the page points
  to for Blackwell's tensor cores).
* same page §5.1: redundant copies of high-load experts from the load
  statistics; §1.3 / §5.1 expert parallelism: the receive side's regrouping
  of rows from source order into expert order.

The page's formulas were lost in extraction; each step below restates the
prose.  Readings where the pages are silent (tie-breaks, the "at the mean"
case, the fp32 sigmoid op sequence needed for bit-exact selection) are marked
READING and listed in the design notes.

Precision: the expert FFN, the router logits and the layer output are fp64
arithmetic on the exact values of the bf16 / fp32 inputs.  Routing decisions
(sigmoid, bias add, group sums, top-K, gate division) are taken in fp32, in
the exact IEEE operation order written here, because floating point decides
an index there and both sides must take that decision in the same precision.

Parity status: every function here is pinned by a ``-m "not gpu"`` test
(closed forms, brute force on tiny inputs, invariants the pages state,
finite differences, and textbook reductions) -- see tests/test_oracle_pins.py,
test_oracle_margin_pins.py, test_oracle_balance_pins.py,
test_oracle_fp8_pins.py, test_oracle_mx_pins.py,
test_oracle_backward_pins.py, test_oracle_expert_backward_pins.py,
test_oracle_ep_pins.py and test_planner.py.
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32

# --------------------------------------------------------------------------
# Spec S1 -- the fp32 sigmoid used for selection (READING R7).
#
# sigma(z) = 1 / (1 + e^{-z}).  The pages fix no rounding; bit-exact routing
# needs one fixed sequence of correctly-rounded IEEE fp32 operations:
#   w = min(max(-z, -32), 80)           (fmax/fmin: NaN z -> -32)
#   n = rint(w * LOG2E)                 (round half to even)
#   r = (w - n*LN2_HI) - n*LN2_LO       (Cody & Waite 1980 two-part ln 2)
#   p = Horner of the degree-7 Taylor polynomial of e^r, each step one
#       rounded multiply then one rounded add (no fused multiply-add)
#   e = p * 2^n                         (exact: the clamp keeps it normal)
#   s = 1 / (1 + e)                     (rounded add, rounded divide)
# For w < -32, e^w < 2^-46 so 1 + e rounds to 1 and the clamp changes
# nothing; w > 80 (z < -80) is clamped (s stays a normal number).
# The constants are derived here from the mathematics (double precision
# ln 2 and factorials), not taken from any library.
# --------------------------------------------------------------------------
_LN2 = math.log(2.0)
LN2_HI = F32(round(_LN2 * 2 ** 16) / 2 ** 16)  # 16 significant bits
LN2_LO = F32(_LN2 - float(LN2_HI))
LOG2E = F32(1.0 / _LN2)
TAYLOR = [F32(1.0 / math.factorial(k)) for k in range(8)]  # 1/k!, k = 0..7


def sig32(z: np.ndarray) -> np.ndarray:
    """fp32 sigmoid by spec S1 (elementwise, any shape)."""
    z = np.asarray(z, dtype=F32)
    w = np.fmin(np.fmax(-z, F32(-32.0)), F32(80.0))
    n = np.rint(w * LOG2E)                      # fp32 multiply, then rint
    r = (w - n * LN2_HI) - n * LN2_LO           # n*LN2_HI is exact
    p = np.full_like(r, TAYLOR[7])
    for k in range(6, -1, -1):
        p = p * r + TAYLOR[k]                   # two rounded fp32 ops
    two_n = ((n.astype(np.int32) + 127) << 23).view(F32)
    e = p * two_n
    return F32(1.0) / (F32(1.0) + e)


# --------------------------------------------------------------------------
# Router logits (eq. 15 context: the affinity is the sigmoid of a token's
# score against each expert's router vector).
# --------------------------------------------------------------------------
def router_logits(x_f32: np.ndarray, w_router: np.ndarray,
                  offset: np.ndarray | None = None) -> np.ndarray:
    """z[t, e] = fl32( sum_h x[t,h] * W_r[e,h] + o[e] ), summed in fp64,
    rounded once (the affinity's argument, §1.3 eq. 15).

    ``x_f32`` holds the exact values of the bf16 activations.  ``offset``
    o[E] is an optional additive term of the router's linear map: V3's
    router has none (o = 0); the skewed-load workload puts its per-expert
    preference there."""
    z = np.asarray(x_f32, np.float64) @ np.asarray(w_router, np.float64).T
    if offset is not None:
        z = z + np.asarray(offset, np.float64)[None, :]
    return z.astype(F32)


# --------------------------------------------------------------------------
# Routing: sigmoid + bias, group limit, top-K, gates (§1.3, §1.4).
# --------------------------------------------------------------------------
def route(logits: np.ndarray, bias: np.ndarray, n_group: int,
          topk_group: int, topk: int, group_on_unbiased: bool = False):
    """Selection and gates for every token.

    Returns dict with
      idx[T,K] int32  -- chosen experts, slot k = k-th by (u desc, e asc)
      gate[T,K] fp32  -- s_{e_k} / sum_j s_{e_j} (raw affinity, never u)
      s[T,E], u[T,E] fp32, group_score[T,G] fp32, kept[T,G] bool

    Steps (all fp32, in this order):
      s = sig32(z); u = s + b                     (eq. 15, eq. 16)
      S_g = u_(1) + u_(2) over the group's two largest u (duplicates count
            twice)                                (§1.3, K_r/M = 2)
      kept = first topk_group groups by (S_g desc, g asc)   READING R3
      idx  = first topk experts of kept groups by (u desc, e asc)
      den  = s_{e_0} + ... + s_{e_{K-1}}, left to right in slot order
      gate = s_{e_k} / den                        (eq. 13)
    ``group_on_unbiased`` scores groups on s instead of u (ablation only;
    the default follows the reading that group limiting is part of the
    biased selection condition, READING R2).
    """
    z = np.asarray(logits, F32)
    T, E = z.shape
    assert E % n_group == 0 and E // n_group >= 2
    assert 1 <= topk_group <= n_group and topk <= topk_group * (E // n_group)
    s = sig32(z)
    u = s + np.asarray(bias, F32)[None, :]

    gs = E // n_group
    grp_vals = (s if group_on_unbiased else u).reshape(T, n_group, gs)
    two = -np.sort(-grp_vals, axis=2)[:, :, :2]      # two largest, multiset
    group_score = two[:, :, 0] + two[:, :, 1]        # fp32 add

    gorder = np.argsort(-group_score, axis=1, kind="stable")[:, :topk_group]
    kept = np.zeros((T, n_group), bool)
    np.put_along_axis(kept, gorder, True, axis=1)

    expert_kept = np.repeat(kept, gs, axis=1)
    cand = np.where(expert_kept, u, F32(-np.inf))
    idx = np.argsort(-cand, axis=1, kind="stable")[:, :topk].astype(np.int32)

    sk = np.take_along_axis(s, idx, axis=1)
    den = np.zeros(T, F32)
    for k in range(topk):                            # slot order, fp32
        den = den + sk[:, k]
    gate = sk / den[:, None]
    return dict(idx=idx, gate=gate.astype(F32), s=s, u=u,
                group_score=group_score, kept=kept)


def routing_margins(r: dict, topk_group: int, topk: int):
    """Per-token decision margins on the oracle's own fp32 u / S:
    top-K margin  u_(K) - u_(K+1) among the kept experts, and
    group margin  S_(M) - S_(M+1) (inf when every group is kept).
    Tokens with small margins may legitimately route differently when the
    logits differ by fp32 rounding (tolerance scope, READING R11)."""
    u = r["u"].astype(np.float64)
    T, E = u.shape
    G = r["group_score"].shape[1]
    kept_e = np.repeat(r["kept"], E // G, axis=1)
    cand = np.sort(np.where(kept_e, u, -np.inf), axis=1)[:, ::-1]
    km = cand[:, topk - 1] - cand[:, topk] if topk < cand.shape[1] else \
        np.full(T, np.inf)
    km = np.where(np.isfinite(km), km, np.inf)
    S = np.sort(r["group_score"].astype(np.float64), axis=1)[:, ::-1]
    gm = S[:, topk_group - 1] - S[:, topk_group] if topk_group < G else \
        np.full(T, np.inf)
    return km, gm


# --------------------------------------------------------------------------
# Load histogram and the stable permutation (dispatch order).
# --------------------------------------------------------------------------
def expert_counts(idx: np.ndarray, E: int) -> np.ndarray:
    """c_e = #{(t, k) : idx[t, k] == e}  (the batch load, §1.4)."""
    return np.bincount(np.asarray(idx).ravel(), minlength=E).astype(np.int32)


def permutation(idx: np.ndarray, E: int):
    """Stable counting sort of the (token, slot) pairs by expert.

    offsets[0] = 0, offsets[e+1] = offsets[e] + c_e
    dest[t, k] = offsets[e] + #{t' < t : e chosen by t'}   (READING R10)
    src_row[dest[t, k]] = t*K + k
    A token chooses an expert at most once, so ordering flat positions
    p = t*K + k is ordering by token inside each expert."""
    idx = np.asarray(idx)
    T, K = idx.shape
    c = expert_counts(idx, E)
    offsets = np.zeros(E + 1, np.int32)
    offsets[1:] = np.cumsum(c)
    order = np.argsort(idx.ravel(), kind="stable")
    dest = np.empty(T * K, np.int32)
    dest[order] = np.arange(T * K, dtype=np.int32)
    return dict(offsets=offsets, dest=dest.reshape(T, K),
                src_row=order.astype(np.int32), counts=c)


# --------------------------------------------------------------------------
# Expert FFN and the layer output (§1.1, eq. 12).
# --------------------------------------------------------------------------
def silu(v: np.ndarray) -> np.ndarray:
    """silu(v) = v / (1 + e^{-v}) in fp64.  For v below about -709, e^{-v}
    overflows to inf and the quotient is the correct limit -0."""
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def swiglu_ffn(a: np.ndarray, w1: np.ndarray, w3: np.ndarray,
               w2: np.ndarray) -> np.ndarray:
    """y = W2 (silu(W1 a) * (W3 a)) for each row a, all fp64, no rounding of
    the intermediate.  w1, w3: [I, H]; w2: [H, I] (values, any float dtype)."""
    a = np.asarray(a, np.float64)
    p = a @ np.asarray(w1, np.float64).T
    q = a @ np.asarray(w3, np.float64).T
    return (silu(p) * q) @ np.asarray(w2, np.float64).T


def moe_output(x: np.ndarray, ys: np.ndarray, y_slots: np.ndarray,
               gate: np.ndarray) -> np.ndarray:
    """out_t = x_t + ys_t + sum_{k=0..K-1} g_{t,k} * y_{e_k}(t)   (eq. 12),
    fp64, summed in slot order.  y_slots[t, k, :] is FFN_{e_k}(x_t)."""
    out = np.asarray(x, np.float64) + np.asarray(ys, np.float64)
    for k in range(y_slots.shape[1]):
        out = out + np.asarray(gate[:, k], np.float64)[:, None] * y_slots[:, k]
    return out


def layer_forward(x_f32, w_router, bias, w1, w3, w2, ws1, ws3, ws2, *,
                  n_group, topk_group, topk):
    """Full layer for every token (small sizes).  Weight arguments hold the
    values (fp32 or fp64 arrays): w1, w3 [E,I,H], w2 [E,H,I]; ws* shared.

    Returns dict: out[T,H] fp64, logits, the routing dict, ys, y_slots."""
    x64 = np.asarray(x_f32, np.float64)
    z = router_logits(x_f32, w_router)
    r = route(z, bias, n_group, topk_group, topk)
    T, K = r["idx"].shape
    E = w1.shape[0]
    ys = swiglu_ffn(x64, ws1, ws3, ws2)
    y_slots = np.zeros((T, K, x64.shape[1]))
    for e in range(E):
        t, k = np.nonzero(r["idx"] == e)
        if t.size:
            y_slots[t, k] = swiglu_ffn(x64[t], w1[e], w3[e], w2[e])
    out = moe_output(x64, ys, y_slots, r["gate"])
    return dict(out=out, logits=z, route=r, ys=ys, y_slots=y_slots)


def layer_rows(x_rows_f32, idx_rows, gate_rows, expert_w, shared_w):
    """Layer output for a sample of tokens whose routing is already known
    (used to check sampled outputs at full V3 size).

    expert_w(e) -> (w1[I,H], w3[I,H], w2[H,I]) values; shared_w likewise."""
    x64 = np.asarray(x_rows_f32, np.float64)
    ys = swiglu_ffn(x64, *shared_w)
    n, K = idx_rows.shape
    y_slots = np.zeros((n, K, x64.shape[1]))
    for e in np.unique(idx_rows):
        t, k = np.nonzero(idx_rows == e)
        y_slots[t, k] = swiglu_ffn(x64[t], *expert_w(int(e)))
    return moe_output(x64, ys, y_slots, gate_rows)


# --------------------------------------------------------------------------
# Auxiliary-loss-free bias update (§1.4).
# --------------------------------------------------------------------------
def bias_update(counts: np.ndarray, bias: np.ndarray, T: int, K: int,
                gamma: float, tie_overloaded: bool = False):
    """One end-of-step update on the whole batch's load.

    Expert e is overloaded when c_e > T*K/E and underloaded when c_e < T*K/E
    (compared exactly as c_e*E vs T*K in integers); b_e -= gamma resp.
    b_e += gamma in fp32 with gamma = fl32(gamma).  An expert exactly at the
    mean is left unchanged (READING R4; ``tie_overloaded`` instead treats
    it as overloaded).  Returns (new_bias, (max, mean, min) load)."""
    c = np.asarray(counts, np.int64)
    b = np.asarray(bias, F32)
    E = c.shape[0]
    g = F32(gamma)
    lhs = c * E
    rhs = np.int64(T) * np.int64(K)
    over = lhs >= rhs if tie_overloaded else lhs > rhs
    under = lhs < rhs
    nb = np.where(over, b - g, np.where(under, b + g, b)).astype(F32)
    stats = (float(c.max()) if E else 0.0, float(T * K) / E if E else 0.0,
             float(c.min()) if E else 0.0)
    return nb, stats


# --------------------------------------------------------------------------
# Sequence-wise balance loss (§1.4, eq. 17-20): the small complementary
# loss kept beside the bias, alpha = 1e-4 for V3.
# --------------------------------------------------------------------------
def seq_balance_loss(logits: np.ndarray, seq_len: int, topk: int,
                     alpha: float = 1e-4):
    """Forward value of the sequence-wise balance loss, one per sequence.

    The batch's T tokens are cut into sequences of ``seq_len`` consecutive
    tokens; the last one holds the remainder (READING R16).  For a sequence
    of T_s tokens and E routed experts:
      s      = sig32(z)                      the affinity, as in routing
      s'_t,i = s_t,i / sum_j s_t,j           (eq. 19, normalised affinity)
      P_i    = (1/T_s) sum_t s'_t,i          (eq. 20)
      f_i    = E / (topk * T_s) * #{t : i among the topk largest s_t}
                                             (eq. 18; raw s -- no bias, no
                                             group limit; ties: lower index)
      L      = alpha * sum_i f_i P_i         (eq. 17)
    The top-K decision is taken on the fp32 s (bit-exact on both sides);
    s', P, f and L are fp64 from those fp32 values.

    Returns dict with counts[n_seq, E] int32 (the indicator sums), f and P
    [n_seq, E] fp64 and loss[n_seq] fp64."""
    z = np.asarray(logits, F32)
    T, E = z.shape
    assert seq_len >= 1 and 1 <= topk <= E
    n_seq = -(-T // seq_len)
    s = sig32(z)
    top = np.argsort(-s, axis=1, kind="stable")[:, :topk]
    chosen = np.zeros((T, E), bool)
    np.put_along_axis(chosen, top, True, axis=1)
    s64 = s.astype(np.float64)
    sp = s64 / s64.sum(axis=1, keepdims=True)
    counts = np.zeros((n_seq, E), np.int32)
    P = np.zeros((n_seq, E))
    f = np.zeros((n_seq, E))
    loss = np.zeros(n_seq)
    for q in range(n_seq):
        a, b = q * seq_len, min(T, (q + 1) * seq_len)
        Ts = b - a
        counts[q] = chosen[a:b].sum(axis=0)
        P[q] = sp[a:b].sum(axis=0) / Ts
        f[q] = E * counts[q].astype(np.float64) / (topk * Ts)
        loss[q] = alpha * float(np.dot(f[q], P[q]))
    return dict(counts=counts, P=P, f=f, loss=loss)


# --------------------------------------------------------------------------
# FP8 (E4M3) fine-grained quantization ("02 · DeepSeek-V3" §2, mixed
# precision): activations grouped in 1 x 128 tiles (one token, 128
# channels), weights in 128 x 128 blocks, one scale per group from the
# group's own max |value| taken online, every tensor in E4M3 (4 exponent
# bits, 3 mantissa bits).
# --------------------------------------------------------------------------
E4M3_MAX = 448.0           # 1.75 * 2^8, the largest finite E4M3 value
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_SUB_STEP = 2.0 ** -9  # spacing of the subnormals


def e4m3_decode(code: np.ndarray) -> np.ndarray:
    """Value of each E4M3 code (uint8): sign bit, 4-bit exponent with bias
    7, 3-bit mantissa; exponent 0 holds the subnormals m/8 * 2^-6; the
    all-ones pattern (exponent 15, mantissa 7) is NaN; no infinities."""
    c = np.asarray(code, np.uint8).astype(np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, m / 8.0 * E4M3_MIN_NORMAL,
                   (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return s * mag


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Round each fp32 value to the nearest E4M3 value, ties to the even
    mantissa, magnitudes beyond 448 saturated to 448 (READING R19: the
    "satfinite" conversion); the sign of a zero result is kept.  Finite
    inputs only."""
    x = np.asarray(x, F32).astype(np.float64)
    assert np.all(np.isfinite(x))
    neg = np.signbit(x)
    a = np.abs(x)
    _, k = np.frexp(np.maximum(a, E4M3_MIN_NORMAL))   # a = f 2^k, f in [.5,1)
    step = np.where(a < E4M3_MIN_NORMAL, E4M3_SUB_STEP, np.exp2(k - 4.0))
    q = np.minimum(np.rint(a / step) * step, E4M3_MAX)  # rint: half to even
    # encode the (exactly representable) magnitude q
    _, kq = np.frexp(np.maximum(q, E4M3_MIN_NORMAL))
    sub = q < E4M3_MIN_NORMAL
    ebits = np.where(sub, 0, kq - 1 + 7)
    mbits = np.where(sub, np.rint(q / E4M3_SUB_STEP),
                     np.rint(q / np.exp2(kq - 1.0) * 8.0) - 8.0)
    code = (neg.astype(np.int64) << 7) | (ebits.astype(np.int64) << 3) | \
        mbits.astype(np.int64)
    return code.astype(np.uint8)


def _group_scale(amax: np.ndarray) -> np.ndarray:
    """scale = fl32(amax / 448); an all-zero group gets scale 1 (READING
    R20), so its codes are all zero either way."""
    amax = np.asarray(amax, F32)
    return np.where(amax > 0, amax / F32(E4M3_MAX), F32(1.0)).astype(F32)


def quantize_1x128(x: np.ndarray):
    """Activation quantization: x [R, C] fp32 (C % 128 == 0) -> codes
    [R, C] uint8 and scales [R, C/128] fp32.  Per row and 128-channel tile:
    amax = max |x|, s = fl32(amax / 448), code = E4M3(fl32(x / s))."""
    x = np.asarray(x, F32)
    R, C = x.shape
    assert C % 128 == 0
    t = x.reshape(R, C // 128, 128)
    s = _group_scale(np.abs(t).max(axis=2))
    q = e4m3_encode((t / s[:, :, None]).astype(F32))
    return q.reshape(R, C), s


def quantize_128x128(w: np.ndarray):
    """Weight quantization: w [R, C] fp32 (both multiples of 128) -> codes
    [R, C] uint8 and scales [R/128, C/128] fp32, one scale per 128 x 128
    block from the block's max |w|."""
    w = np.asarray(w, F32)
    R, C = w.shape
    assert R % 128 == 0 and C % 128 == 0
    b = w.reshape(R // 128, 128, C // 128, 128)
    s = _group_scale(np.abs(b).max(axis=(1, 3)))
    q = e4m3_encode((b / s[:, None, :, None]).astype(F32))
    return q.reshape(R, C), s


def dequantize(q: np.ndarray, s: np.ndarray, rows_per_scale: int):
    """Exact value of quantized data in fp64: code value x its group's
    scale (rows_per_scale = 1 for 1x128 tiles, 128 for 128x128 blocks)."""
    v = e4m3_decode(q)
    sc = np.repeat(np.repeat(np.asarray(s, np.float64), rows_per_scale,
                             axis=0), 128, axis=1)
    return v * sc


def fp8_swiglu_ffn(a_q, a_s, w1, w3, w2, requant=None):
    """One expert on FP8 inputs (§2 mixed precision on §1.1's SwiGLU):
    a_q / a_s the 1x128-quantized token rows; w1, w3, w2 each a
    (codes, scales) pair of 128x128-quantized weights.
      p, q = A W1^T, A W3^T on the dequantized values (fp64, exact
             products: the pages' full-precision accumulation)
      m    = silu(p) * q, rounded to fp32, then 1x128-quantized
             (READING R21: the down projection's input is FP8 too) by
             `requant` (quantize_1x128 unless given: the power-of-two
             variant passes quantize_1x128_pow2)
      y    = M W2^T on the dequantized values (fp64)
    Returns y (fp64) and the intermediate (codes, scales)."""
    requant = quantize_1x128 if requant is None else requant
    A = dequantize(a_q, a_s, 1)
    p = A @ dequantize(*w1, 128).T
    q = A @ dequantize(*w3, 128).T
    m = (silu(p) * q).astype(F32)
    m_q, m_s = requant(m)
    y = dequantize(m_q, m_s, 1) @ dequantize(*w2, 128).T
    return y, (m_q, m_s)


# --------------------------------------------------------------------------
# The same groups with power-of-two scales.  The pages (same page, §2) liken
# the fine-grained groups to the microscaling formats whose scaling
# Blackwell's tensor cores apply natively; in those formats a group's scale
# is a power of two, stored as an 8-bit biased exponent (UE8M0).  READING
# R28: with power-of-two scales the group scale is the least power of two
# that keeps the group's largest magnitude within 448, i.e. 2^e with e the
# least integer such that 448 * 2^e >= amax (clamped below at -127, the
# smallest UE8M0 exponent; an all-zero group gets e = 0), and every code is
# the E4M3 rounding of the exact quotient x / 2^e.
# --------------------------------------------------------------------------
UE8M0_BIAS = 127


def group_exponent_pow2(amax: np.ndarray) -> np.ndarray:
    """e = min{integer e : 448 * 2^e >= amax}, at least -127; 0 when
    amax == 0.  From the definition: a floating estimate of log2(amax/448),
    then exact corrections (448 * 2^e is exact in fp64)."""
    a = np.asarray(amax, F32).astype(np.float64)
    pos = a > 0
    est = np.where(pos, np.ceil(np.log2(np.where(pos, a, 1.0) / E4M3_MAX)),
                   0.0).astype(np.int64)
    for _ in range(2):
        est = np.where(pos & (np.ldexp(E4M3_MAX, est) < a), est + 1, est)
        est = np.where(pos & (np.ldexp(E4M3_MAX, est - 1) >= a), est - 1,
                       est)
    assert np.all(~pos | (np.ldexp(E4M3_MAX, est) >= a))
    assert np.all(~pos | (np.ldexp(E4M3_MAX, est - 1) < a))
    return np.where(pos, np.maximum(est, -UE8M0_BIAS), 0)


def ue8m0_encode(e: np.ndarray) -> np.ndarray:
    """The scale 2^e as its UE8M0 byte e + 127."""
    return (np.asarray(e, np.int64) + UE8M0_BIAS).astype(np.uint8)


def ue8m0_decode(b: np.ndarray) -> np.ndarray:
    """The scale of a UE8M0 byte: 2^(b - 127) (fp32; byte 255 is not a
    scale this quantizer writes)."""
    return np.ldexp(1.0, np.asarray(b, np.int64) - UE8M0_BIAS).astype(F32)


def _codes_pow2(t: np.ndarray, e: np.ndarray) -> np.ndarray:
    # x / 2^e is exact in fp64; rounded to fp32 it changes only below
    # 2^-126, where the E4M3 code is 0 either way
    return e4m3_encode(np.ldexp(t.astype(np.float64), -e).astype(F32))


def quantize_1x128_pow2(x: np.ndarray):
    """quantize_1x128 with power-of-two scales: codes [R, C] uint8 and
    scales [R, C/128] fp32 (each 2^e, e from group_exponent_pow2)."""
    x = np.asarray(x, F32)
    R, C = x.shape
    assert C % 128 == 0
    t = x.reshape(R, C // 128, 128)
    e = group_exponent_pow2(np.abs(t).max(axis=2))
    q = _codes_pow2(t, e[:, :, None])
    return q.reshape(R, C), ue8m0_decode(ue8m0_encode(e))


def quantize_128x128_pow2(w: np.ndarray):
    """quantize_128x128 with power-of-two scales: codes [R, C] uint8 and
    scales [R/128, C/128] fp32 (each 2^e)."""
    w = np.asarray(w, F32)
    R, C = w.shape
    assert R % 128 == 0 and C % 128 == 0
    b = w.reshape(R // 128, 128, C // 128, 128)
    e = group_exponent_pow2(np.abs(b).max(axis=(1, 3)))
    q = _codes_pow2(b, e[:, None, :, None])
    return q.reshape(R, C), ue8m0_decode(ue8m0_encode(e))


# --------------------------------------------------------------------------
# Expert parallelism's receive side ("02 · DeepSeek-V3" §1.3, node-limited
# routing over experts partitioned across devices; §5.1, the EP deployment):
# the rows a device receives arrive source by source, each source's rows
# sorted by expert ("source-major"); the grouped GEMM wants each local
# expert's rows together, sources in order ("expert-major").
# --------------------------------------------------------------------------
def ep_plan(recv_counts: np.ndarray):
    """recv_counts [P, El]: rows source s sends for local expert l.
    Source-major row order: (s, l, j) sorted by s, then l, then j;
    expert-major: by l, then s, then j.  Returns (perm [rows], offsets
    [El + 1]): perm[i] = expert-major position of source-major row i;
    offsets[l] = first expert-major row of local expert l."""
    rc = np.asarray(recv_counts, np.int64)
    P, El = rc.shape
    rows = int(rc.sum())
    # first row of block (s, l) in each order: counts before it, row-major
    # (source-major) resp. column-major (expert-major)
    src_first = (np.cumsum(rc.ravel()) - rc.ravel()).reshape(P, El)
    exp_first = (np.cumsum(rc.T.ravel()) - rc.T.ravel()).reshape(El, P).T
    perm = np.empty(rows, np.int64)
    for s in range(P):
        for l in range(El):
            n = int(rc[s, l])
            a = int(src_first[s, l])
            perm[a:a + n] = exp_first[s, l] + np.arange(n)
    offsets = np.append(exp_first[0, :], rows)
    return perm, offsets


# --------------------------------------------------------------------------
# Redundant-expert planning from the load histogram ("02 · DeepSeek-V3"
# §5.1: high-load experts are replicated from online load statistics, e.g.
# 32 redundant experts with one extra expert per GPU, and the set is
# revised periodically).
# --------------------------------------------------------------------------
def plan_redundant_experts(load: np.ndarray, n_devices: int,
                           slots_per_device: int):
    """Place up to R = n_devices * slots_per_device redundant expert copies
    (READING R24).

    Base placement: device d hosts experts [d*E/D, (d+1)*E/D); its load is
    the sum of their loads.  An expert with a copy serves its c tokens
    round-robin: the original keeps ceil(c/2), the copy floor(c/2).
    Walk the experts heaviest first (load desc, index asc) while slots are
    free and loads are positive; an expert gets a copy on the device with
    the smallest current load among those with a free slot other than its
    own (ties: lower device); an expert whose only free slots are on its own
    device is passed over.
    Returns dict: slot_expert [D, slots] int32 (-1 = empty slot),
    device_load [D] int64 after planning, base_load [D] int64 before,
    replicated: the experts given a copy, in placement order."""
    c = np.asarray(load, np.int64)
    E = c.shape[0]
    D, r = int(n_devices), int(slots_per_device)
    assert D >= 1 and r >= 0 and E % D == 0
    per = E // D
    dev = np.array([c[d * per:(d + 1) * per].sum() for d in range(D)],
                   np.int64)
    base = dev.copy()
    slots = [[] for _ in range(D)]
    free = D * r
    placed = []
    for e in sorted(range(E), key=lambda q: (-c[q], q)):
        if free == 0 or c[e] <= 0:
            break
        home = e // per
        cand = [d for d in range(D) if len(slots[d]) < r and d != home]
        if not cand:
            continue
        d = min(cand, key=lambda q: (dev[q], q))
        share = c[e] // 2
        dev[home] -= share
        dev[d] += share
        slots[d].append(e)
        placed.append(e)
        free -= 1
    slot_expert = np.full((D, r), -1, np.int32)
    for d in range(D):
        slot_expert[d, :len(slots[d])] = slots[d]
    return dict(slot_expert=slot_expert, device_load=dev, base_load=base,
                replicated=np.array(placed, np.int32))


# --------------------------------------------------------------------------
# Backward of routing to the router logits (the training-side neighbour of
# §1.4): the gates' and the balance loss's gradients.  The top-K choices
# and the balance loss's indicator counts are piecewise constant in z, so
# they carry no gradient (READING R25); the bias is not in backpropagation
# (the pages say so).  s = sig32(z) as in the forward; the rest in fp64.
# --------------------------------------------------------------------------
def route_backward(logits: np.ndarray, idx: np.ndarray,
                   dgate: np.ndarray) -> np.ndarray:
    """dL/dz from the gates' upstream gradient dgate [T, K].
    g_k = s_k / D with D = sum of the chosen s; for a chosen expert m:
      dL/dz_m = s_m (1 - s_m) / D * (dgate_m - sum_k dgate_k g_k)
    and 0 for the experts not chosen.  Returns [T, E] fp64."""
    z = np.asarray(logits, F32)
    T, E = z.shape
    s = sig32(z).astype(np.float64)
    idx = np.asarray(idx)
    dg = np.asarray(dgate, np.float64)
    sk = np.take_along_axis(s, idx, axis=1)
    D = sk.sum(axis=1, keepdims=True)
    g = sk / D
    dot = (dg * g).sum(axis=1, keepdims=True)
    out = np.zeros((T, E))
    np.put_along_axis(out, idx, sk * (1 - sk) / D * (dg - dot), axis=1)
    return out


def seq_balance_loss_backward(logits: np.ndarray, seq_len: int, topk: int,
                              alpha: float = 1e-4, dloss=None) -> np.ndarray:
    """dL/dz of the sequence-wise balance loss (eq. 17-20), L per sequence
    times its upstream gradient dloss[q] (default 1).  With S_t = sum_j
    s_t,j, s' = s / S_t and f from the forward's counts:
      dL/dz_t,i = dloss_q * alpha / T_s * s_i (1 - s_i) / S_t
                  * (f_i - sum_j f_j s'_t,j)
    Returns [T, E] fp64."""
    z = np.asarray(logits, F32)
    T, E = z.shape
    fw = seq_balance_loss(z, seq_len, topk, alpha)
    n_seq = fw["loss"].shape[0]
    dl = np.ones(n_seq) if dloss is None else np.asarray(dloss, np.float64)
    s = sig32(z).astype(np.float64)
    S = s.sum(axis=1, keepdims=True)
    out = np.zeros((T, E))
    for q in range(n_seq):
        a, b = q * seq_len, min(T, (q + 1) * seq_len)
        f = fw["f"][q]
        sp = s[a:b] / S[a:b]
        dot = sp @ f
        out[a:b] = dl[q] * alpha / (b - a) * s[a:b] * (1 - s[a:b]) / S[a:b] \
            * (f[None, :] - dot[:, None])
    return out


# --------------------------------------------------------------------------
# Backward of the experts and of the combine (§1.1 SwiGLU, eq. 12), fp64.
# --------------------------------------------------------------------------
def swiglu_ffn_backward(a, w1, w3, w2, dy):
    """Gradients of y = W2 (silu(W1 a) * (W3 a)) for rows a [n, H], given
    dy [n, H]; with p = a W1^T, q = a W3^T, m = silu(p) q:
      dm  = dy W2            dW2 = dy^T m
      dq  = dm silu(p)       dp  = dm q silu'(p),
                             silu'(p) = sigma(p) (1 + p (1 - sigma(p)))
      dW1 = dp^T a           dW3 = dq^T a
      da  = dp W1 + dq W3
    Returns (da [n, H], dw1 [I, H], dw3 [I, H], dw2 [H, I])."""
    a = np.asarray(a, np.float64)
    w1, w3, w2 = (np.asarray(w, np.float64) for w in (w1, w3, w2))
    dy = np.asarray(dy, np.float64)
    p = a @ w1.T
    q = a @ w3.T
    sg = 1.0 / (1.0 + np.exp(-p))
    m = p * sg * q
    dm = dy @ w2
    dw2 = dy.T @ m
    dq = dm * p * sg
    dp = dm * q * sg * (1.0 + p * (1.0 - sg))
    return dp @ w1 + dq @ w3, dp.T @ a, dq.T @ a, dw2


def combine_backward(dout, y_slots, gate):
    """Gradients of out_t = x_t + ys_t + sum_k g_{t,k} y_{t,k} (eq. 12):
    dx_t (residual) = dys_t = dout_t, dy_{t,k} = g_{t,k} dout_t and
    dgate_{t,k} = <dout_t, y_{t,k}> (the input of route_backward).
    Returns (dx_residual, dys, dy_slots [T, K, H], dgate [T, K])."""
    d = np.asarray(dout, np.float64)
    y = np.asarray(y_slots, np.float64)
    g = np.asarray(gate, np.float64)
    return d, d, g[:, :, None] * d[:, None, :], np.einsum("th,tkh->tk", d, y)


def layer_backward(x, dout, idx, gate, w1, w3, w2, ws1, ws3, ws2):
    """Backward of the layer's expert part for a fixed routing (§1.1 SwiGLU
    experts, eq. 12 combine), fp64, from the pinned pieces above.

    out_t = x_t + FFN_s(x_t) + sum_k g_{t,k} FFN_{e_k}(x_t)   (eq. 12)
    Given dout [T, H]:
      dgate[t, k] = <dout_t, FFN_{e_k}(x_t)>                (combine_backward)
      dx_t        = dout_t + dFFN_s(x_t)^T dout_t
                    + sum_k dFFN_{e_k}(x_t)^T (g_{t,k} dout_t)
                    (residual, shared and routed experts; the path through
                    the router's logits is route_backward's, not this one)
      dW*_e       = swiglu_ffn_backward over the rows routed to e, with the
                    upstream gradient g_{t,k} dout_t; the shared expert's
                    over all tokens with dout_t.
    Weight arguments hold values: w1, w3 [E, I, H], w2 [E, H, I]; ws*
    shared.  Returns dict(dx [T, H], dgate [T, K], dw1, dw3 [E, I, H],
    dw2 [E, H, I], dws1, dws3 [I_s, H], dws2 [H, I_s])."""
    x64 = np.asarray(x, np.float64)
    d = np.asarray(dout, np.float64)
    idx = np.asarray(idx)
    g = np.asarray(gate, np.float64)
    T, K = idx.shape
    E = w1.shape[0]
    dxs, dws1, dws3, dws2 = swiglu_ffn_backward(x64, ws1, ws3, ws2, d)
    dx = d + dxs
    dgate = np.zeros((T, K))
    dw1 = np.zeros(np.shape(w1))
    dw3 = np.zeros(np.shape(w3))
    dw2 = np.zeros(np.shape(w2))
    for e in range(E):
        t, k = np.nonzero(idx == e)
        if t.size == 0:
            continue
        a = x64[t]
        y = swiglu_ffn(a, w1[e], w3[e], w2[e])
        dgate[t, k] = np.einsum("nh,nh->n", d[t], y)
        da, dw1[e], dw3[e], dw2[e] = swiglu_ffn_backward(
            a, w1[e], w3[e], w2[e], g[t, k][:, None] * d[t])
        dx[t] += da          # a token chooses an expert at most once
    return dict(dx=dx, dgate=dgate, dw1=dw1, dw3=dw3, dw2=dw2, dws1=dws1,
                dws3=dws3, dws2=dws2)
