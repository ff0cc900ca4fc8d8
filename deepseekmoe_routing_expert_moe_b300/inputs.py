"""Seeded synthetic inputs for the DeepSeekMoE layer forward.

This module is the one piece that both the CUDA path's tests/bench and the CPU
oracle consume.  It holds NO arithmetic of the method: it only draws random
numbers, rounds them to bf16 storage, and lays them out.  Every tensor is keyed
by (config seed, tensor id, expert, step) through numpy's ``SeedSequence`` so
any single expert's weights can be regenerated on the host without touching
the others (the oracle uses that to check sampled tokens at full V3 size).

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
    "decode_v3": MoEConfig("decode_v3", 3, T=128, H=7168, E=256, n_group=8,
                           topk_group=4, topk=8, I=2048, I_shared=2048),
    "skewed_v3": MoEConfig("skewed_v3", 4, T=32768, H=7168, E=256, n_group=8,
                           topk_group=4, topk=8, I=2048, I_shared=2048,
                           zipf_s=1.2, zipf_beta=1.0, steps=50),
}


def custom_config(name: str, config_id: int, **kw) -> MoEConfig:
    """A config with its own seed space (for parity sweeps over shapes)."""
    return MoEConfig(name, config_id, **kw)


def _rng(cfg: MoEConfig, tensor: str, expert: int = 0, step: int = 0):
    ss = np.random.SeedSequence([BASE_SEED + cfg.config_id, _TID[tensor],
                                 expert, step])
    return np.random.Generator(np.random.PCG64(ss))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Storage rounding: fp32 -> bf16 bit pattern, round to nearest even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def _normal_bf16(rng, shape, sigma):
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        a *= np.float32(sigma)
    return f32_to_bf16_bits(a)


# ----------------------------------------------------------------- activations
def x_tokens(cfg: MoEConfig, step: int = 0, T: int | None = None) -> np.ndarray:
    """Activations x[T, H] ~ N(0, 1), bf16 bits."""
    T = cfg.T if T is None else T
    return _normal_bf16(_rng(cfg, "x", 0, step), (T, cfg.H), 1.0)


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
def expert_weights(cfg: MoEConfig, e: int):
    """Routed expert e: (w1[I,H], w3[I,H], w2[H,I]) bf16 bits ~ N(0, w_sigma)."""
    s = cfg.w_sigma
    return (_normal_bf16(_rng(cfg, "w1", e), (cfg.I, cfg.H), s),
            _normal_bf16(_rng(cfg, "w3", e), (cfg.I, cfg.H), s),
            _normal_bf16(_rng(cfg, "w2", e), (cfg.H, cfg.I), s))


def shared_weights(cfg: MoEConfig):
    """Shared expert: (ws1[I_s,H], ws3[I_s,H], ws2[H,I_s]) bf16 bits."""
    s = cfg.w_sigma
    return (_normal_bf16(_rng(cfg, "ws1"), (cfg.I_shared, cfg.H), s),
            _normal_bf16(_rng(cfg, "ws3"), (cfg.I_shared, cfg.H), s),
            _normal_bf16(_rng(cfg, "ws2"), (cfg.H, cfg.I_shared), s))


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


def stream_expert_weights(cfg: MoEConfig, sink, threads: int | None = None):
    """Generate routed experts one at a time and hand each to ``sink(e, w1,
    w3, w2)`` (used to fill device memory without holding all 22.5 GB of the
    V3 layer on the host)."""
    with ThreadPoolExecutor(threads or os.cpu_count() or 4) as ex:
        for e, ws in enumerate(ex.map(lambda i: expert_weights(cfg, i),
                                      range(cfg.E))):
            sink(e, *ws)


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
