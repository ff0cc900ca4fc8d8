"""The C ABI without a GPU: the library loads, exports every entry point
include/moe.h declares, sizes workspaces, and rejects bad arguments on the
host before anything is launched (only failing calls are made here)."""
import ctypes
import os
import re

import pytest

from deepseekmoe_routing_expert_moe_b300 import build, ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return ops.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_six_layer_entry_points():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_combine",
              "moe_bias_update", "moe_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    # and the binding wraps each under the same name
    for n in names:
        assert n in ops._SIGS, n


def test_abi_version_and_status_strings(L):
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        want = int(re.search(r"#define MOE_ABI_VERSION (\d+)", f.read())[1])
    assert want == 4 and ops.moe_abi_version() == want


def test_build_entry_point_checks_the_built_library(L):
    """__graft_entry__.build() compiles and verifies the library's
    interface version against the header (run here without a GPU)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "graft_entry", os.path.join(ROOT, "__graft_entry__.py"))
    g = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(g)
    g.build()
    for code, name in ops.STATUS.items():
        assert ops.moe_status_string(code) == name


V3 = dict(T=4096, H=7168, E=256, n_group=8, topk_group=4, topk=8, I=2048,
          I_shared=2048, gamma=0.001)


def test_workspace_sizes_are_consistent(L):
    d = ops.dims(**V3)
    r = ops.workspace_bytes(d, ops.MOE_WS_ROUTE)
    p = ops.workspace_bytes(d, ops.MOE_WS_PERMUTE)
    f = ops.workspace_bytes(d, ops.MOE_WS_EXPERT_FFN)
    fw = ops.workspace_bytes(d, ops.MOE_WS_FORWARD)
    assert 0 < r <= fw and 0 < p <= fw and 0 < f <= fw
    # the forward workspace holds xp, yp (T*K*H bf16 each) and h at 128
    # rows per expert (at decode the up GEMM gathers the rows from x)
    assert fw >= 2 * 4096 * 8 * 7168 * 2 + 4096 * 8 * 2048 * 2
    dd = ops.dims(**dict(V3, T=128))
    fd = ops.workspace_bytes(dd, ops.MOE_WS_FORWARD)
    assert 128 * 8 * 7168 * 2 + 128 * 8 * 2048 * 2 <= fd
    bad = ops.dims(**dict(V3, E=255))
    assert ops.workspace_bytes(bad, ops.MOE_WS_FORWARD) == 0
    assert ops.workspace_bytes(d, 9) == 0


FAKE = 1 << 20  # a 16-byte aligned address; never dereferenced here


def _route(L, d, ws_bytes=1 << 30, logits=FAKE, ws=FAKE):
    return L.moe_route(ctypes.byref(d), logits, FAKE, FAKE, FAKE, FAKE, ws,
                       ws_bytes, None)


@pytest.mark.parametrize("over,code", [
    (dict(E=255), 1),            # E % n_group != 0
    (dict(n_group=4, topk_group=5), 1),
    (dict(topk=33, topk_group=8), 2),
    (dict(E=16, n_group=16, topk_group=2, topk=2), 1),  # group of 1
    (dict(T=-1), 1),
    (dict(topk=0), 1),
    (dict(topk=129), 1),         # more than topk_group * group size
    (dict(E=48, n_group=8, topk_group=4, topk=8), 2),   # E % 32
    (dict(E=2048, n_group=32, topk_group=4, topk=8), 2),
    (dict(H=7000), 2),
    (dict(E=96, n_group=8, topk_group=4, topk=8), 2),   # 3 experts per lane
    (dict(gamma=float("nan")), 1),
    (dict(T=(1 << 31) // 9 + 1), 2),   # T*(topk+1) rows overflow int32
])
def test_route_rejects_bad_dims(L, over, code):
    d = ops.dims(**dict(V3, **over))
    assert _route(L, d) == code


def test_null_misaligned_and_small_workspace(L):
    d = ops.dims(**V3)
    assert _route(L, d, logits=None) == 1
    assert _route(L, d, logits=FAKE + 4) == 3
    assert _route(L, d, ws=None) == 4
    assert _route(L, d, ws_bytes=16) == 4
    assert L.moe_route(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30,
                       None) == 1


def test_ffn_and_forward_validation(L):
    d = ops.dims(**V3)
    w = ops.MoeWeights(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None)
    assert L.moe_expert_ffn(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE,
                            FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == 1
    w = ops.MoeWeights(FAKE, FAKE, FAKE, FAKE + 2, FAKE, FAKE, FAKE)
    assert L.moe_expert_ffn(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE,
                            FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == 3
    d2 = ops.dims(**dict(V3, I=100))
    w = ops.MoeWeights(*(FAKE,) * 7)
    assert L.moe_forward(ctypes.byref(d2), ctypes.byref(w), FAKE, FAKE, 0,
                         FAKE, None, None, None, None, None, FAKE, 1 << 40,
                         None) == 2
    assert L.moe_forward(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE, 0,
                         FAKE, None, None, None, None, None, FAKE, 100,
                         None) == 4
    assert L.moe_combine(ctypes.byref(d), FAKE, FAKE, None, FAKE, FAKE, FAKE,
                         None) == 1
    assert L.moe_bias_update(ctypes.byref(d), FAKE, None, None, None) == 1
    assert L.moe_permute(ctypes.byref(d), None, FAKE, FAKE, FAKE, FAKE, FAKE,
                         FAKE, 1 << 30, None) == 1
    assert L.moe_get_device_error(None, None) == 1
    # the optional router offset must be 16-byte aligned too
    w = ops.MoeWeights(*(FAKE,) * 7, FAKE + 4)
    assert L.moe_forward(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE, 0,
                         FAKE, None, None, None, None, None, FAKE, 1 << 40,
                         None) == 3
    assert L.moe_router_logits(ctypes.byref(d), FAKE, FAKE, FAKE + 8, FAKE,
                               FAKE, 1 << 40, None) == 3
    # ... and so must the optional prepared router split
    w = ops.MoeWeights(*(FAKE,) * 7, None, FAKE + 2)
    assert L.moe_forward(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE, 0,
                         FAKE, None, None, None, None, None, FAKE, 1 << 40,
                         None) == 3


def test_router_weight_split_validation(L):
    rs = L.moe_router_weight_split
    assert rs(FAKE, 0, 7168, FAKE, None) == 1
    assert rs(FAKE, 256, 0, FAKE, None) == 1
    assert rs(FAKE, 200, 7168, FAKE, None) == 2       # E % 16: no split
    assert rs(None, 256, 7168, FAKE, None) == 1
    assert rs(FAKE, 256, 7168, None, None) == 1
    assert rs(FAKE + 4, 256, 7168, FAKE, None) == 3
    assert rs(FAKE, 256, 7168, FAKE + 8, None) == 3


def _balance(L, d, seq_len=4096, alpha=1e-4, logits=FAKE, out=FAKE,
             ws=FAKE, ws_bytes=1 << 30):
    return L.moe_seq_balance_loss(ctypes.byref(d), logits, seq_len, alpha,
                                  out, FAKE, FAKE, ws, ws_bytes, None)


def test_seq_balance_validation_and_workspace(L):
    d = ops.dims(**V3)
    need = ops.workspace_bytes(d, ops.MOE_WS_SEQ_BALANCE)
    # s' (fp32) and the top-K flags (u8) for every token and expert
    assert need >= 4096 * 256 * 5
    assert need <= ops.workspace_bytes(d, ops.MOE_WS_FORWARD)
    # a forward workspace covers it even where the layer's own buffers are
    # small next to [T, E] (many experts, narrow hidden size)
    wide = ops.dims(**dict(V3, H=64, E=1024, n_group=32, topk=1,
                           topk_group=1, I=64, I_shared=64))
    assert 0 < ops.workspace_bytes(wide, ops.MOE_WS_SEQ_BALANCE) <= \
        ops.workspace_bytes(wide, ops.MOE_WS_FORWARD)
    assert _balance(L, d, seq_len=0) == 1
    assert _balance(L, d, seq_len=-5) == 1
    assert _balance(L, d, alpha=float("nan")) == 1
    assert _balance(L, d, alpha=float("inf")) == 1
    assert _balance(L, d, logits=None) == 1
    assert _balance(L, d, out=None) == 1
    assert _balance(L, d, out=FAKE + 4) == 3
    assert _balance(L, d, ws_bytes=need - 1) == 4
    assert _balance(L, ops.dims(**dict(V3, E=255))) == 1
    # no tokens: nothing to compute, nothing launched, NULL tensors allowed
    d0 = ops.dims(**dict(V3, T=0))
    assert L.moe_seq_balance_loss(ctypes.byref(d0), None, 7, 1e-4, None, None,
                                  None, FAKE, 1 << 20, None) == 0


def test_fp8_quantization_validation(L):
    qb, qr = L.moe_quantize_fp8_blocks, L.moe_quantize_fp8_rows
    assert qb(FAKE, 100, 128, FAKE, FAKE, None) == 1       # rows % 128
    assert qb(FAKE, 128, 100, FAKE, FAKE, None) == 1       # cols % 128
    assert qb(FAKE, 128 * 65536, 128, FAKE, FAKE, None) == 2
    assert qb(None, 128, 128, FAKE, FAKE, None) == 1
    assert qb(FAKE, 128, 128, FAKE + 4, FAKE, None) == 3
    assert qb(FAKE, 0, 128, None, None, None) == 0         # nothing to do
    assert qr(FAKE, 5, 100, FAKE, FAKE, None) == 1
    assert qr(FAKE, -1, 128, FAKE, FAKE, None) == 1
    assert qr(FAKE, 5, 128, FAKE, FAKE + 8, None) == 3
    assert qr(FAKE, 0, 128, None, None, None) == 0
    d = ops.dims(**V3)
    pf = L.moe_permute_fp8

    def call(dd, x=FAKE, dest=FAKE, xps=FAKE, ws_bytes=1 << 30):
        return pf(ctypes.byref(dd), x, dest, FAKE, FAKE, FAKE, xps, FAKE,
                  ws_bytes, None)
    assert call(d, dest=None) == 1
    assert call(d, xps=FAKE + 8) == 3
    assert call(d, ws_bytes=16) == 4
    assert call(ops.dims(**dict(V3, H=192))) == 2           # H % 128
    assert pf(ctypes.byref(ops.dims(**dict(V3, T=0))), None, None, None,
              None, None, None, FAKE, 1 << 30, None) == 0


def test_fp8_ffn_validation(L):
    d = ops.dims(**V3)
    fn = L.moe_expert_ffn_fp8
    need = ops.workspace_bytes(d, ops.MOE_WS_EXPERT_FFN_FP8)
    # E4M3 intermediate codes + scales for the routed and the shared rows
    assert need >= 4096 * 8 * 2048 + 4096 * 2048
    assert need <= ops.workspace_bytes(d, ops.MOE_WS_FORWARD)

    def call(dd, w, xs=FAKE, ws_bytes=1 << 40):
        return fn(ctypes.byref(dd), ctypes.byref(w), FAKE, FAKE, FAKE, xs,
                  FAKE, FAKE, FAKE, FAKE, ws_bytes, None)
    good = ops.MoeWeightsFp8(*(FAKE,) * 12)
    assert call(ops.dims(**dict(V3, H=192)), good) == 2      # H % 128
    assert call(ops.dims(**dict(V3, I=64 * 3)), good) == 2   # I % 128
    assert call(ops.dims(**dict(V3, H=8192 + 128)), good) == 2
    assert call(d, ops.MoeWeightsFp8(*(FAKE,) * 11, None)) == 1
    assert call(d, ops.MoeWeightsFp8(*(FAKE,) * 5, FAKE + 4,
                                     *(FAKE,) * 6)) == 3
    assert call(d, good, xs=FAKE + 8) == 3
    assert call(d, good, ws_bytes=1024) == 4
    d0 = ops.dims(**dict(V3, T=0))
    assert fn(ctypes.byref(d0), ctypes.byref(good), None, None, None, None,
              FAKE, None, None, FAKE, 1 << 20, None) == 0


def test_mx_quantization_validation(L):
    qb, qr = L.moe_quantize_mx_blocks, L.moe_quantize_mx_rows
    assert qb(FAKE, 100, 128, FAKE, FAKE, None) == 1       # rows % 128
    assert qb(FAKE, 128, 100, FAKE, FAKE, None) == 1       # cols % 128
    assert qb(FAKE, 128 * 65536, 128, FAKE, FAKE, None) == 2
    assert qb(FAKE, 128, 128, FAKE, None, None) == 1
    assert qb(FAKE, 128, 128, FAKE, FAKE + 4, None) == 3
    assert qb(FAKE, 0, 128, None, None, None) == 0         # nothing to do
    assert qr(FAKE, 5, 100, FAKE, FAKE, None) == 1
    assert qr(FAKE, -1, 128, FAKE, FAKE, None) == 1
    assert qr(FAKE + 2, 5, 128, FAKE, FAKE, None) == 3
    assert qr(FAKE, 0, 128, None, None, None) == 0
    d = ops.dims(**V3)
    pm = L.moe_permute_mx

    def call(dd, x=FAKE, dest=FAKE, xps=FAKE, ws_bytes=1 << 30):
        return pm(ctypes.byref(dd), x, dest, FAKE, FAKE, FAKE, xps, FAKE,
                  ws_bytes, None)
    assert call(d, x=None) == 1
    assert call(d, xps=FAKE + 8) == 3
    assert call(d, ws_bytes=16) == 4
    assert call(ops.dims(**dict(V3, H=192))) == 2           # H % 128
    assert pm(ctypes.byref(ops.dims(**dict(V3, T=0))), None, None, None,
              None, None, None, FAKE, 1 << 30, None) == 0


def test_mx_ffn_validation(L):
    d = ops.dims(**V3)
    fn = L.moe_expert_ffn_mx
    need = ops.workspace_bytes(d, ops.MOE_WS_EXPERT_FFN_MX)
    # E4M3 intermediate codes + UE8M0 scales, routed and shared rows
    assert need >= 4096 * 8 * 2048 * (1 + 1 / 128) + 4096 * 2048
    assert need <= ops.workspace_bytes(d, ops.MOE_WS_FORWARD)

    def call(dd, w, xs=FAKE, ws_bytes=1 << 40):
        return fn(ctypes.byref(dd), ctypes.byref(w), FAKE, FAKE, FAKE, xs,
                  FAKE, FAKE, FAKE, FAKE, ws_bytes, None)
    good = ops.MoeWeightsMx(*(FAKE,) * 12)
    assert call(ops.dims(**dict(V3, H=192)), good) == 2      # H % 128
    assert call(ops.dims(**dict(V3, I=64 * 3)), good) == 2   # I % 128
    assert call(d, ops.MoeWeightsMx(*(FAKE,) * 11, None)) == 1
    assert call(d, ops.MoeWeightsMx(*(FAKE,) * 5, FAKE + 4,
                                    *(FAKE,) * 6)) == 3
    assert call(d, good, xs=FAKE + 8) == 3
    assert call(d, good, ws_bytes=1024) == 4
    d0 = ops.dims(**dict(V3, T=0))
    assert fn(ctypes.byref(d0), ctypes.byref(good), None, None, None, None,
              FAKE, None, None, FAKE, 1 << 20, None) == 0


def test_routing_backward_validation(L):
    d = ops.dims(**V3)
    rb, bb = L.moe_route_backward, L.moe_seq_balance_loss_backward
    by = ctypes.byref
    assert rb(by(d), FAKE, None, FAKE, 0, FAKE, FAKE, 1 << 30, None) == 1
    assert rb(by(d), FAKE, FAKE, FAKE + 4, 0, FAKE, FAKE, 1 << 30, None) == 3
    assert rb(by(d), FAKE, FAKE, FAKE, 0, FAKE, FAKE, 8, None) == 4
    assert rb(by(ops.dims(**dict(V3, T=0))), None, None, None, 0, None,
              FAKE, 1 << 20, None) == 0
    assert bb(by(d), FAKE, 0, 1e-4, FAKE, None, 0, FAKE, None) == 1
    assert bb(by(d), FAKE, 64, float("nan"), FAKE, None, 0, FAKE,
              None) == 1
    assert bb(by(d), FAKE, 64, 1e-4, None, None, 0, FAKE, None) == 1
    assert bb(by(d), FAKE, 64, 1e-4, FAKE, FAKE + 4, 0, FAKE, None) == 3
    assert bb(by(ops.dims(**dict(V3, T=0))), None, 64, 1e-4, None, None, 0,
              None, None) == 0
    fb = L.moe_route_balance_backward

    def fused(dd=d, logits=FAKE, idx=FAKE, dg=FAKE, S=64, alpha=1e-4,
              counts=FAKE, dloss=None, out=FAKE, ws_bytes=1 << 30):
        return fb(by(dd), logits, idx, dg, S, alpha, counts, dloss, 0, out,
                  FAKE, ws_bytes, None)
    assert fused(idx=None) == 1
    assert fused(counts=None) == 1
    assert fused(S=0) == 1
    assert fused(alpha=float("inf")) == 1
    assert fused(dloss=FAKE + 4) == 3
    assert fused(dg=FAKE + 2) == 3
    assert fused(ws_bytes=8) == 4
    assert fused(dd=ops.dims(**dict(V3, E=255))) == 1
    assert fused(dd=ops.dims(**dict(V3, T=0)), logits=None, idx=None,
                 dg=None, counts=None, out=None, ws_bytes=1 << 20) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(ops, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(ops, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        ops.lib()


def test_expert_backward_validation(L):
    d = ops.dims(**V3)
    fn = L.moe_expert_backward
    by = ctypes.byref
    need = ops.workspace_bytes(d, ops.MOE_WS_EXPERT_BWD)
    # padded dispatch rows (T*K + 15*E) of x, dout, the recomputed p, q
    # (fp32) and the dgrad rows
    cap = 4096 * 8 + 15 * 256
    assert need >= cap * 7168 * 2 * 3 + cap * 2048 * 4 * 2
    w = ops.MoeWeights(*(FAKE,) * 7, None)

    def call(dd=d, ww=w, x=FAKE, dw1=FAKE, ws_bytes=1 << 40):
        return fn(by(dd), by(ww), x, FAKE, FAKE, FAKE, 0, FAKE, FAKE, dw1,
                  FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws_bytes, None)
    assert call(x=None) == 1
    assert call(dw1=None) == 1
    assert call(ww=ops.MoeWeights(FAKE, None, *(FAKE,) * 5, None)) == 1
    assert call(x=FAKE + 2) == 3
    assert call(ws_bytes=4096) == 4
    assert call(dd=ops.dims(**dict(V3, I=100))) == 2


def test_routed_ffn_and_expert_parallel_maps_validation(L):
    by = ctypes.byref
    # no routing here: one expert, one group is fine
    d1 = ops.dims(T=100, H=256, E=1, n_group=1, topk_group=1, topk=1, I=128,
                  I_shared=64)
    assert ops.workspace_bytes(d1, ops.MOE_WS_EXPERT_FFN) > 0
    assert ops.workspace_bytes(d1, ops.MOE_WS_ROUTE) == 0   # routing rules
    w = ops.MoeWeights(None, FAKE, FAKE, FAKE, None, None, None, None)
    fr = L.moe_expert_ffn_routed
    assert fr(by(d1), by(w), FAKE, FAKE, FAKE, FAKE, 8, None) == 4
    assert fr(by(d1), by(ops.MoeWeights(None, None, FAKE, FAKE, None, None,
                                        None, None)),
              FAKE, FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert fr(by(ops.dims(T=100, H=250, E=1, n_group=1, topk_group=1,
                          topk=1, I=128, I_shared=64)), by(w), FAKE, FAKE,
              FAKE, FAKE, 1 << 30, None) == 2
    plan, rows = L.moe_ep_plan, L.moe_ep_permute_rows
    assert plan(0, 4, FAKE, 10, FAKE, FAKE, None, None) == 1
    assert plan(65, 64, FAKE, 10, FAKE, FAKE, None, None) == 2  # > 4096 cells
    assert plan(2, 4, FAKE, -1, FAKE, FAKE, None, None) == 1
    assert plan(2, 4, FAKE + 4, 10, FAKE, FAKE, None, None) == 3
    assert rows(FAKE, 10, 0, FAKE, 0, FAKE, None, None) == 1    # width
    assert rows(FAKE, 10, 32, None, 0, FAKE, None, None) == 1
    assert rows(FAKE + 8, 10, 32, FAKE, 0, FAKE, None, None) == 3
    assert rows(None, 0, 32, None, 0, None, None, None) == 0
    # the FP8 (power-of-two) routed experts: the same dims rules, widths
    # multiples of 128, NULL shared weights allowed
    d2 = ops.dims(T=100, H=256, E=1, n_group=1, topk_group=1, topk=1, I=128,
                  I_shared=128)
    assert ops.workspace_bytes(d2, ops.MOE_WS_EXPERT_FFN_MX) > 0
    wm = ops.MoeWeightsMx(*(FAKE,) * 6, *(None,) * 6)
    fm = L.moe_expert_ffn_mx_routed
    assert fm(by(d2), by(wm), FAKE, FAKE, FAKE, FAKE, FAKE, 8, None) == 4
    assert fm(by(d2), by(ops.MoeWeightsMx(*(FAKE,) * 5, None, *(None,) * 6)),
              FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert fm(by(d2), by(wm), FAKE, FAKE + 4, FAKE, FAKE, FAKE, 1 << 30,
              None) == 3
    assert fm(by(ops.dims(T=100, H=192, E=1, n_group=1, topk_group=1,
                          topk=1, I=128, I_shared=128)), by(wm), FAKE, FAKE,
              FAKE, FAKE, FAKE, 1 << 30, None) == 2
    d0 = ops.dims(T=0, H=256, E=1, n_group=1, topk_group=1, topk=1, I=128,
                  I_shared=128)
    assert fm(by(d0), by(wm), None, None, FAKE, None, FAKE, 1 << 20,
              None) == 0
