"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random numbers: it holds none of the layer's
arithmetic (no routing, quantisation, dispatch, GEMM or combine), so both the
CUDA path and the CPU oracle can take their inputs from it.  Every tensor is
drawn from its own ``torch.Generator`` on the requested device, seeded from
(seed, layer, tensor id, sub-index), so any piece can be regenerated alone.
Values are drawn in fp32 and rounded to bf16 by ``Tensor.to`` (round to
nearest even).  The same seed gives different numbers on CPU and CUDA.

Workloads (shapes and distributions of the large-MoE setting that the
prime-rl "RL at 1T Scale" post trains with router replay and block-scaled
FP8; the post prints no data, so all inputs are synthetic):

  tiny               T=256,  d=256,  E=8,   k=2, F=512,  softmax top-k routing
  replay             T=4096, d=2048, E=64,  k=6, F=1408, replayed ids, Zipf(1.1)
  large              T=8192, d=7168, E=256, k=8, F=2048, sigmoid top-k routing
  long_dispatch      T=131072, d=7168, E=256, k=8, identity experts (bf16 rows)
  multilayer_replay  8 layers x T=16384 at the large shape, skewed replayed ids
  large_e64          T=2048, d=7168, E=64, k=8, F=2048 (profiling size of "large")
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

SOFTMAX = 0
SIGMOID = 1

# tensor ids for seeding
_X, _WR, _W13, _W2, _IDS, _GATES, _PERM = 1, 2, 3, 4, 5, 6, 7


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int            # tokens
    d: int            # hidden size
    E: int            # experts
    k: int            # top_k
    F: int            # expert FFN size (SwiGLU: W13 has 2F rows)
    score_fn: int     # SOFTMAX or SIGMOID
    mode: str         # "route" (router top-k), "replay" (payload ids), "identity"
    ids_dist: str     # "router" | "zipf" | "uniform" | "hot_cold"
    w_std: float = 0.02
    wr_std: float = 0.02
    layers: int = 1
    renorm: int = 1
    route_scale: float = 1.0
    zipf_s: float = 1.1
    hot_frac: float = 0.3
    n_hot: int = 8
    n_cold: int = 8

    @property
    def A(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


CONFIGS = {
    "tiny": MoEConfig("tiny", 256, 256, 8, 2, 512, SOFTMAX, "route", "router", w_std=0.02),
    "replay": MoEConfig("replay", 4096, 2048, 64, 6, 1408, SOFTMAX, "replay", "zipf", w_std=0.02),
    "large": MoEConfig("large", 8192, 7168, 256, 8, 2048, SIGMOID, "route", "router", w_std=0.006),
    "long_dispatch": MoEConfig("long_dispatch", 131072, 7168, 256, 8, 2048, SIGMOID, "identity",
                               "uniform", w_std=0.006),
    "multilayer_replay": MoEConfig("multilayer_replay", 16384, 7168, 256, 8, 2048, SIGMOID, "replay",
                                   "hot_cold", w_std=0.006, layers=8),
    # profiling shape: the large layer's per-expert GEMM shape (about 256 rows
    # per expert, d=7168, F=2048) with a quarter of the experts and tokens, so
    # that a profiler capture holds ~3.5 GB instead of ~14 GB
    "large_e64": MoEConfig("large_e64", 2048, 7168, 64, 8, 2048, SIGMOID, "route", "router", w_std=0.006),
    # weight-gradient profiling shape: the same per-expert shape with 16
    # experts, so that dW13 [16, 4096, 7168] and dW2 [16, 7168, 2048] fp32
    # hold ~2.8 GB
    "large_e16": MoEConfig("large_e16", 512, 7168, 16, 8, 2048, SIGMOID, "route", "router", w_std=0.006),
}


def _gen(device, seed: int, layer: int, tensor: int, sub: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((((seed * 128 + layer) * 16 + tensor) << 16) + sub)
    return g


def _normal_bf16(shape, std, g, device) -> torch.Tensor:
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def make_x(cfg: MoEConfig, device, seed: int = 0, layer: int = 0, T: int | None = None) -> torch.Tensor:
    """x ~ N(0, 1), bf16 [T, d]."""
    T = cfg.T if T is None else T
    return _normal_bf16((T, cfg.d), 1.0, _gen(device, seed, layer, _X), device)


def make_router_w(cfg: MoEConfig, device, seed: int = 0, layer: int = 0) -> torch.Tensor:
    """W_r ~ N(0, wr_std), bf16 [E, d]."""
    return _normal_bf16((cfg.E, cfg.d), cfg.wr_std, _gen(device, seed, layer, _WR), device)


def make_w13_expert(cfg: MoEConfig, e: int, device, seed: int = 0, layer: int = 0) -> torch.Tensor:
    """Expert e's fused gate/up weight ~ N(0, w_std), bf16 [2F, d] (rows 0..F-1 gate, F..2F-1 up)."""
    return _normal_bf16((2 * cfg.F, cfg.d), cfg.w_std, _gen(device, seed, layer, _W13, e), device)


def make_w2_expert(cfg: MoEConfig, e: int, device, seed: int = 0, layer: int = 0) -> torch.Tensor:
    """Expert e's down weight ~ N(0, w_std), bf16 [d, F]."""
    return _normal_bf16((cfg.d, cfg.F), cfg.w_std, _gen(device, seed, layer, _W2, e), device)


def make_w13(cfg: MoEConfig, device, seed: int = 0, layer: int = 0) -> torch.Tensor:
    out = torch.empty((cfg.E, 2 * cfg.F, cfg.d), dtype=torch.bfloat16, device=device)
    for e in range(cfg.E):
        out[e] = make_w13_expert(cfg, e, device, seed, layer)
    return out


def make_w2(cfg: MoEConfig, device, seed: int = 0, layer: int = 0) -> torch.Tensor:
    out = torch.empty((cfg.E, cfg.d, cfg.F), dtype=torch.bfloat16, device=device)
    for e in range(cfg.E):
        out[e] = make_w2_expert(cfg, e, device, seed, layer)
    return out


def _distinct_by_keys(keys: torch.Tensor, k: int) -> torch.Tensor:
    """Indices of the k largest keys per row, in descending key order (a
    Gumbel-top-k draw when keys = log p + Gumbel noise)."""
    return torch.argsort(keys, dim=1, descending=True, stable=True)[:, :k]


def _gumbel(shape, g, device) -> torch.Tensor:
    u = torch.rand(shape, generator=g, device=device, dtype=torch.float64)
    u = u.clamp_min(1e-300)
    return -torch.log(-torch.log(u).clamp_min(1e-300))


def make_replay_payload(cfg: MoEConfig, device, seed: int = 0) -> torch.Tensor:
    """Routed-experts payload int32 [layers, k, T]: ids a token was routed to
    at inference, slot order = draw order, k distinct ids per token.

    zipf:     expert popularity p(rank r) ~ r^-s (r = 1..E), rank -> expert
              through a seeded permutation; k distinct per token by
              Gumbel-top-k (= sequential sampling without replacement).
    uniform:  k distinct uniformly at random.
    hot_cold: per layer a seeded hot set H (n_hot experts) and cold set Z
              (n_cold experts that receive no tokens); each slot is hot with
              probability hot_frac (uniform over H minus those taken), else
              uniform over the experts outside H and Z minus those taken.
    """
    T, k, E = cfg.T, cfg.k, cfg.E
    out = torch.empty((cfg.layers, k, T), dtype=torch.int32, device=device)
    for l in range(cfg.layers):
        g = _gen(device, seed, l, _IDS)
        if cfg.ids_dist == "zipf":
            perm = torch.randperm(E, generator=_gen(device, seed, l, _PERM), device=device)
            ranks = torch.arange(1, E + 1, device=device, dtype=torch.float64)
            logp_rank = -cfg.zipf_s * torch.log(ranks)
            logp = torch.empty(E, dtype=torch.float64, device=device)
            logp[perm] = logp_rank
            ids = _distinct_by_keys(logp[None, :] + _gumbel((T, E), g, device), k)
        elif cfg.ids_dist == "uniform":
            ids = _distinct_by_keys(torch.rand((T, E), generator=g, device=device), k)
        elif cfg.ids_dist == "hot_cold":
            perm = torch.randperm(E, generator=_gen(device, seed, l, _PERM), device=device)
            hot = perm[: cfg.n_hot]
            rest = perm[cfg.n_hot + cfg.n_cold:]
            hot_mask = torch.rand((T, k), generator=g, device=device) < cfg.hot_frac
            hot_pick = hot[_distinct_by_keys(torch.rand((T, cfg.n_hot), generator=g, device=device), k)
                           if k <= cfg.n_hot else
                           _distinct_by_keys(torch.rand((T, cfg.n_hot), generator=g, device=device), cfg.n_hot)]
            rest_pick = rest[_distinct_by_keys(torch.rand((T, rest.numel()), generator=g, device=device), k)]
            hot_rank = torch.cumsum(hot_mask.to(torch.int64), dim=1) - 1
            rest_rank = torch.cumsum((~hot_mask).to(torch.int64), dim=1) - 1
            hot_rank = hot_rank.clamp(0, hot_pick.shape[1] - 1)
            rest_rank = rest_rank.clamp(0, k - 1)
            ids = torch.where(hot_mask, torch.gather(hot_pick, 1, hot_rank), torch.gather(rest_pick, 1, rest_rank))
        else:
            raise ValueError(f"no payload distribution for {cfg.ids_dist!r}")
        out[l] = ids.t().to(torch.int32)
    return out


def make_dirichlet_gates(cfg: MoEConfig, device, seed: int = 0) -> torch.Tensor:
    """Gates ~ Dirichlet(1) over the k slots: Exp(1) draws normalised per
    token, fp32 [T, k]."""
    g = _gen(device, seed, 0, _GATES)
    u = torch.rand((cfg.T, cfg.k), generator=g, device=device, dtype=torch.float64).clamp_min(1e-300)
    e = -torch.log(u)
    return (e / e.sum(dim=1, keepdim=True)).to(torch.float32)
