"""Seeded synthetic inputs for the DeepSeekMoE layer forward.

This module is the one piece that both the CUDA path's tests/bench and the CPU
oracle consume.  It holds NO arithmetic of the method: it only draws random
numbers, rounds them to bf16 storage, and lays them out.

bf16 tensors (activations and expert weights) come from a counter-based
generator: element i of a tensor with 32-bit key k (derived by numpy's
``SeedSequence`` from config seed, tensor id, expert and step) gets the
16-bit cell  mix32(i * 0x9E3779B1 + k) & 0xFFFF,  where mix32 is a
multiply/xor-shift finaliser whose multipliers are below 2^31, so every
intermediate fits in a signed 64-bit integer without overflow.  The cell
picks one of 2^16 equiprobable cells of N(0, sigma); the value is that
cell's midpoint quantile, rounded to bf16 (inverse-transform sampling from
the normal quantised to 2^16 cells, support +-4.3 sigma, finer than bf16).
The same integer formula runs in numpy on the host and in torch on the GPU
and gives identical bits, so the 22.5 GB of V3 expert weights are generated
directly in device memory while the oracle regenerates any single expert on
the host.  fp32 tensors (router weight, bias, logits) are small and are
drawn on the host from Philox streams keyed the same way.

Shapes follow the DeepSeek-V3 MoE layer described on "02 · DeepSeek-V3"
(PaperTrace) §1.1 and the walkthrough's config field list ("DeepSeek-V3
架构导读", 配置逐字段解析): hidden 7168, 256 routed experts of intermediate
2048, 1 shared expert, top-8, 8 groups with 4 kept (§1.3).

Storage conventions (shared with the C-ABI):
  * bf16 tensors are numpy ``uint16`` bit patterns (round-to-nearest-even of
    an fp32 draw);
  * routed weights are canonical ``w1[E, I, H]`` (gate), ``w3[E, I, H]`` (up),
    ``w2[E, H, I]`` (down); the shared expert is ``ws1[I_s, H]``,
    ``ws3[I_s, H]``, ``ws2[H, I_s]``;
  * router weight ``w_router[E, H]`` fp32; bias ``b[E]`` fp32.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

BASE_SEED = 20261202

# tensor ids inside one config's seed space
_TID = {"x": 1, "w_router": 2, "w1": 3, "w3": 4, "w2": 5, "ws1": 6, "ws3": 7,
        "ws2": 8, "bias": 9, "zipf_perm": 10, "logits": 11}


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    """One synthetic workload: layer dimensions plus the input recipe."""
    name: str
    config_id: int
    T: int
    H: int
    E: int
    n_group: int
    topk_group: int
    topk: int
    I: int
    I_shared: int
    gamma: float = 0.001
    w_sigma: float = 0.02        # expert weights ~ N(0, w_sigma), bf16
    router_sigma: float = 0.006  # router weight ~ N(0, router_sigma), fp32
    bias_range: float = 0.01     # b ~ U(-bias_range, bias_range)
    zipf_s: float = 0.0          # >0: skewed per-expert logit preference
    zipf_beta: float = 0.0
    steps: int = 1
    weight_seed_id: int = -1     # config whose weights these are (-1: own)

    def dims(self, **over) -> dict:
        d = dict(T=self.T, H=self.H, E=self.E, n_group=self.n_group,
                 topk_group=self.topk_group, topk=self.topk, I=self.I,
                 I_shared=self.I_shared, gamma=self.gamma)
        d.update(over)
        return d


# The five workloads.  Tiny is the case the oracle finishes in seconds.
CONFIGS = {
    "tiny": MoEConfig("tiny", 0, T=64, H=256, E=16, n_group=4, topk_group=2,
                      topk=4, I=64, I_shared=64, router_sigma=0.02),
    "route_v3": MoEConfig("route_v3", 1, T=16384, H=7168, E=256, n_group=8,
                          topk_group=4, topk=8, I=2048, I_shared=2048),
    "prefill_v3": MoEConfig("prefill_v3", 2, T=4096, H=7168, E=256, n_group=8,
                            topk_group=4, topk=8, I=2048, I_shared=2048),
    # decode and the skewed run use the prefill layer's weights and router
    "decode_v3": MoEConfig("decode_v3", 3, T=128, H=7168, E=256, n_group=8,
                           topk_group=4, topk=8, I=2048, I_shared=2048,
                           weight_seed_id=2),
    "skewed_v3": MoEConfig("skewed_v3", 4, T=32768, H=7168, E=256, n_group=8,
                           topk_group=4, topk=8, I=2048, I_shared=2048,
                           zipf_s=1.2, zipf_beta=1.0, steps=50,
                           weight_seed_id=2),
    # profiling stand-in for the prefill layer: the same 128 rows per expert
    # and the same per-expert shapes, but 32 experts (2.9 GB of weights), so
    # that a full counter capture holds only a few GB on the device
    "prefill_v3_e32": MoEConfig("prefill_v3_e32", 5, T=512, H=7168, E=32,
                                n_group=8, topk_group=4, topk=8, I=2048,
                                I_shared=2048),
    # profiling stand-in for the FP8 decode layer: the decode batch (128
    # tokens, top-8) over 32 experts -- 32 rows each, one full token tile --
    # so that the E4M3 weights (1.4 GB) fit a full counter capture
    "decode_v3_e32": MoEConfig("decode_v3_e32", 6, T=128, H=7168, E=32,
                               n_group=8, topk_group=4, topk=8, I=2048,
                               I_shared=2048),
    # profiling stand-in for the experts' backward at the prefill shape:
    # 128 rows per expert as at T = 4096, 16 experts (1.4 GB of weights,
    # 2.8 GB of fp32 weight gradients), so a full counter capture holds a
    # few GB on the device
    "prefill_v3_e16": MoEConfig("prefill_v3_e16", 7, T=256, H=7168, E=16,
                                n_group=4, topk_group=2, topk=8, I=2048,
                                I_shared=2048),
}


def custom_config(name: str, config_id: int, **kw) -> MoEConfig:
    """A config with its own seed space (for parity sweeps over shapes)."""
    return MoEConfig(name, config_id, **kw)


_WEIGHT_TENSORS = ("w_router", "w1", "w3", "w2", "ws1", "ws3", "ws2", "bias")


def _seed_seq(cfg: MoEConfig, tensor: str, expert: int = 0, step: int = 0):
    cid = cfg.config_id
    if tensor in _WEIGHT_TENSORS and cfg.weight_seed_id >= 0:
        cid = cfg.weight_seed_id
    return np.random.SeedSequence([BASE_SEED + cid, _TID[tensor], expert,
                                   step])


def _rng(cfg: MoEConfig, tensor: str, expert: int = 0, step: int = 0):
    return np.random.Generator(np.random.Philox(_seed_seq(cfg, tensor, expert,
                                                          step)))


def _key32(cfg: MoEConfig, tensor: str, expert: int = 0, step: int = 0) -> int:
    return int(_seed_seq(cfg, tensor, expert, step).generate_state(1)[0])


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Storage rounding: fp32 -> bf16 bit pattern, round to nearest even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


_QTABLE: dict = {}


def quantile_table(sigma: float) -> np.ndarray:
    """bf16 bits of sigma * Phi^-1((i + 1/2) / 2^16), i = 0 .. 2^16 - 1."""
    t = _QTABLE.get(sigma)
    if t is None:
        from scipy.special import ndtri
        q = ndtri((np.arange(65536, dtype=np.float64) + 0.5) / 65536.0)
        t = f32_to_bf16_bits((q * sigma).astype(np.float32))
        _QTABLE[sigma] = t
    return t


_GOLD, _MIX1, _MIX2, _M32 = 0x9E3779B1, 0x7FEB352D, 0x2C1B3C6D, 0xFFFFFFFF
_CHUNK = 1 << 24


def cells_numpy(n: int, key: int, start: int = 0) -> np.ndarray:
    """16-bit cells of elements start .. start+n-1, in numpy (a second,
    independent evaluation of the formula; the generator itself runs the
    torch one on the host CPU or the GPU)."""
    x = np.arange(start, start + n, dtype=np.int64)
    x = (x * _GOLD + key) & _M32
    x ^= x >> 16
    x = (x * _MIX1) & _M32
    x ^= x >> 15
    x = (x * _MIX2) & _M32
    x ^= x >> 16
    return (x & 0xFFFF).astype(np.int64)


def cells_torch(n: int, key: int, device, start: int = 0):
    """The same cells computed with torch int64 ops on `device`."""
    import torch
    x = torch.arange(start, start + n, dtype=torch.int64, device=device)
    x = (x * _GOLD + key) & _M32
    x ^= x >> 16
    x = (x * _MIX1) & _M32
    x ^= x >> 15
    x = (x * _MIX2) & _M32
    x ^= x >> 16
    return x & 0xFFFF


def normal_bf16(key: int, shape, sigma: float, device=None):
    """bf16 bits ~ N(0, sigma): numpy uint16 on the host (device=None), or a
    torch int16 tensor generated on `device`; identical bits either way."""
    import torch
    n = int(np.prod(shape))
    table = quantile_table(float(sigma))
    dev = "cpu" if device is None else device
    tab = torch.from_numpy(table.view(np.int16)).to(dev)
    out = torch.empty(n, dtype=torch.int16, device=dev)
    for s0 in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s0)
        out[s0:s0 + m] = tab[cells_torch(m, key, dev, s0)]
    out = out.reshape(shape)
    return out.numpy().view(np.uint16) if device is None else out


# ----------------------------------------------------------------- activations
def x_tokens(cfg: MoEConfig, step: int = 0, T: int | None = None,
             device=None):
    """Activations x[T, H] ~ N(0, 1), bf16 bits (host, or torch on device)."""
    T = cfg.T if T is None else T
    return normal_bf16(_key32(cfg, "x", 0, step), (T, cfg.H), 1.0, device)


def router_weight(cfg: MoEConfig) -> np.ndarray:
    """W_router[E, H] fp32 ~ N(0, router_sigma)."""
    a = _rng(cfg, "w_router").standard_normal(size=(cfg.E, cfg.H),
                                              dtype=np.float32)
    return a * np.float32(cfg.router_sigma)


def bias(cfg: MoEConfig) -> np.ndarray:
    """Initial per-expert bias b[E] fp32 ~ U(-r, r); the skewed run starts at 0."""
    if cfg.zipf_s > 0:
        return np.zeros(cfg.E, np.float32)
    r = cfg.bias_range
    return _rng(cfg, "bias").uniform(-r, r, size=cfg.E).astype(np.float32)


def zipf_preference(cfg: MoEConfig) -> np.ndarray:
    """Per-expert additive logit preference beta * r_e^(-s), r a seeded
    permutation of 1..E (the skewed-load workload); zeros otherwise."""
    if cfg.zipf_s <= 0:
        return np.zeros(cfg.E, np.float32)
    r = _rng(cfg, "zipf_perm").permutation(cfg.E) + 1
    return (cfg.zipf_beta * r.astype(np.float64) ** (-cfg.zipf_s)).astype(
        np.float32)


# --------------------------------------------------------------------- experts
def expert_matrix(cfg: MoEConfig, name: str, e: int, device=None):
    """One matrix ("w1", "w3" [I,H] or "w2" [H,I]) of routed expert e."""
    shape = (cfg.H, cfg.I) if name == "w2" else (cfg.I, cfg.H)
    return normal_bf16(_key32(cfg, name, e), shape, cfg.w_sigma, device)


def expert_weights(cfg: MoEConfig, e: int, device=None):
    """Routed expert e: (w1[I,H], w3[I,H], w2[H,I]) bf16 bits ~ N(0, w_sigma)."""
    return tuple(expert_matrix(cfg, n, e, device) for n in ("w1", "w3", "w2"))


def shared_weights(cfg: MoEConfig, device=None):
    """Shared expert: (ws1[I_s,H], ws3[I_s,H], ws2[H,I_s]) bf16 bits."""
    s = cfg.w_sigma
    return (normal_bf16(_key32(cfg, "ws1"), (cfg.I_shared, cfg.H), s, device),
            normal_bf16(_key32(cfg, "ws3"), (cfg.I_shared, cfg.H), s, device),
            normal_bf16(_key32(cfg, "ws2"), (cfg.H, cfg.I_shared), s, device))


def device_expert_weights(cfg: MoEConfig, device):
    """All routed experts generated in device memory: torch int16 tensors
    w1[E,I,H], w3[E,I,H], w2[E,H,I] (same bits as expert_weights)."""
    import torch
    w1 = torch.empty((cfg.E, cfg.I, cfg.H), dtype=torch.int16, device=device)
    w3 = torch.empty_like(w1)
    w2 = torch.empty((cfg.E, cfg.H, cfg.I), dtype=torch.int16, device=device)
    for e in range(cfg.E):
        w1[e], w3[e], w2[e] = expert_weights(cfg, e, device)
    return w1, w3, w2


def all_expert_weights(cfg: MoEConfig, threads: int | None = None):
    """All routed experts stacked: w1[E,I,H], w3[E,I,H], w2[E,H,I] (host)."""
    w1 = np.empty((cfg.E, cfg.I, cfg.H), np.uint16)
    w3 = np.empty_like(w1)
    w2 = np.empty((cfg.E, cfg.H, cfg.I), np.uint16)

    def fill(e):
        w1[e], w3[e], w2[e] = expert_weights(cfg, e)

    with ThreadPoolExecutor(threads or os.cpu_count() or 4) as ex:
        list(ex.map(fill, range(cfg.E)))
    return w1, w3, w2


def layer_inputs(cfg: MoEConfig, step: int = 0) -> dict:
    """Everything one layer forward needs, on the host (small configs)."""
    w1, w3, w2 = all_expert_weights(cfg)
    ws1, ws3, ws2 = shared_weights(cfg)
    return dict(x=x_tokens(cfg, step), w_router=router_weight(cfg),
                bias=bias(cfg), w1=w1, w3=w3, w2=w2, ws1=ws1, ws3=ws3, ws2=ws2)


def random_logits(cfg: MoEConfig, T: int | None = None, step: int = 0,
                  scale: float = 0.5) -> np.ndarray:
    """Stand-alone fp32 logits ~ N(0, scale) for routing-only edge cases."""
    T = cfg.T if T is None else T
    return (_rng(cfg, "logits", 0, step).standard_normal(
        size=(T, cfg.E), dtype=np.float32) * np.float32(scale))
