"""The seeded input generators give the workloads' structure (distinct ids
per token, skew, zero-token experts, Dirichlet gates) deterministically."""
import numpy as np
import torch

from block_scaled_fp8_router_gb300 import synthetic as S


def _distinct_rows(ids):
    s = np.sort(ids, axis=1)
    return np.all(s[:, 1:] != s[:, :-1])


def test_deterministic():
    cfg = S.CONFIGS["tiny"]
    assert torch.equal(S.make_x(cfg, "cpu"), S.make_x(cfg, "cpu"))
    assert not torch.equal(S.make_x(cfg, "cpu", seed=1), S.make_x(cfg, "cpu"))
    assert torch.equal(S.make_w13_expert(cfg, 3, "cpu"), S.make_w13(cfg, "cpu")[3])


def test_zipf_payload():
    cfg = S.CONFIGS["replay"]
    p = S.make_replay_payload(cfg, "cpu")
    assert p.shape == (1, cfg.k, cfg.T) and p.dtype == torch.int32
    ids = p[0].T.numpy()
    assert ids.min() >= 0 and ids.max() < cfg.E and _distinct_rows(ids)
    c = np.sort(np.bincount(ids.ravel(), minlength=cfg.E))[::-1]
    assert c[0] > 3 * c[cfg.E // 2]          # skewed popularity


def test_hot_cold_payload():
    cfg = S.CONFIGS["multilayer_replay"].with_(T=4096, layers=2)
    p = S.make_replay_payload(cfg, "cpu")
    assert p.shape == (2, 8, 4096)
    for l in range(2):
        ids = p[l].T.numpy()
        assert _distinct_rows(ids)
        c = np.bincount(ids.ravel(), minlength=cfg.E)
        assert (c == 0).sum() == cfg.n_cold
        hot = np.argsort(c)[::-1][: cfg.n_hot]
        frac = c[hot].sum() / c.sum()
        assert 0.27 < frac < 0.33


def test_uniform_payload_and_gates():
    cfg = S.CONFIGS["long_dispatch"].with_(T=2000)
    ids = S.make_replay_payload(cfg, "cpu")[0].T.numpy()
    assert _distinct_rows(ids)
    g = S.make_dirichlet_gates(cfg, "cpu")
    assert g.shape == (2000, 8) and torch.all(g > 0)
    assert torch.allclose(g.double().sum(1), torch.ones(2000, dtype=torch.float64), atol=1e-6)
