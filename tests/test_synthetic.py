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


def test_value_distributions():
    """x ~ N(0, 1), router rows ~ N(0, 0.02), expert weights ~ N(0, w_std)
    (0.02 for the small workloads, 0.006 for the large shapes), all bf16,
    with the layouts the layer takes."""
    for name, w_std in (("tiny", 0.02), ("large", 0.006)):
        cfg = S.CONFIGS[name]
        x = S.make_x(cfg, "cpu", T=512)
        wr = S.make_router_w(cfg, "cpu")
        w13 = S.make_w13_expert(cfg, 1, "cpu")
        w2 = S.make_w2_expert(cfg, 1, "cpu")
        assert x.dtype == wr.dtype == w13.dtype == w2.dtype == torch.bfloat16
        assert x.shape == (512, cfg.d) and wr.shape == (cfg.E, cfg.d)
        assert w13.shape == (2 * cfg.F, cfg.d) and w2.shape == (cfg.d, cfg.F)
        assert cfg.w_std == w_std
        for t, sd in ((x, 1.0), (wr, 0.02), (w13, w_std), (w2, w_std)):
            v = t.double()
            assert abs(v.mean().item()) < 0.05 * sd and abs(v.std().item() / sd - 1) < 0.05, (name, sd)
