"""GPU parity at the full workload sizes, in the launch configuration bench.py
times (the MoELayerFP8 call sequence), against the CPU oracle.

- large (T=8192, d=7168, E=256, top-8, F=2048, sigmoid): router ids of every
  token, gates on a token sample; counts, offsets and both maps in full; the x
  quantisation and the dispatched FP8 rows in full; weight codes of every
  expert; the layer output of every token within the 2e-2 bar.
- long_dispatch (T=131072, d=7168 bf16 rows, E=256, top-8): replay copy and
  maps in full against the oracle; combine(dispatch(x)) == x bit for bit
  with identity experts and Dirichlet gates.
- multilayer_replay (8 layers of the large shape at T=16384, skewed payload
  with zero-token experts): every layer, replay and maps in full, the cold
  experts really empty, and the output on 2048 sampled tokens per layer that
  include a token of every hot expert (rows are independent, so a sample is
  exact).
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_router_gb300 import synthetic as S
from tests.helpers import bf16_bits, bf16_to_f64, row_rel_err

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL = 2e-2


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from block_scaled_fp8_router_gb300 import moe_r3
    return moe_r3


def _layer(cfg, seed=0, layer_idx=0):
    from block_scaled_fp8_router_gb300.layer import MoELayerFP8, MoEWeightsFP8, quantize_weights
    E, d, F = cfg.E, cfg.d, cfg.F
    w = MoEWeightsFP8(S.make_router_w(cfg, DEV, seed, layer_idx),
                      torch.empty((E, 2 * F, d), dtype=torch.uint8, device=DEV),
                      torch.empty((E, 2 * F // 128, d // 128), dtype=torch.float32, device=DEV),
                      torch.empty((E, d, F), dtype=torch.uint8, device=DEV),
                      torch.empty((E, d // 128, F // 128), dtype=torch.float32, device=DEV))
    for e0 in range(0, E, 16):
        n = min(16, E - e0)
        w13 = torch.stack([S.make_w13_expert(cfg, e, DEV, seed, layer_idx) for e in range(e0, e0 + n)])
        w2 = torch.stack([S.make_w2_expert(cfg, e, DEV, seed, layer_idx) for e in range(e0, e0 + n)])
        quantize_weights(w13, w2, out=w, e0=e0)
    return MoELayerFP8(w, cfg.T, cfg.k, cfg.score_fn, cfg.renorm, cfg.route_scale)


def _oracle_tokens(oracle, cfg, layer, tokens, ids, gates_ref, x, seed=0, layer_idx=0):
    """Oracle layer output for the sampled tokens (every expert row they use;
    ids and gates_ref are the sampled tokens' rows), with the oracle's own
    weight quantisation of the experts involved, also checked against the GPU
    codes."""
    k = cfg.k
    used = np.unique(ids)
    remap = {int(e): i for i, e in enumerate(used)}
    w = [[], [], [], []]
    for e in used:
        q, s = oracle.quant_128x128(bf16_bits(S.make_w13_expert(cfg, int(e), DEV, seed, layer_idx)))
        assert np.array_equal(q, layer.w.w13_q[int(e)].cpu().numpy()), f"W13 codes of expert {e}"
        assert np.array_equal(s, layer.w.w13_s[int(e)].cpu().numpy())
        w[0].append(q); w[1].append(s)
        q, s = oracle.quant_128x128(bf16_bits(S.make_w2_expert(cfg, int(e), DEV, seed, layer_idx)))
        assert np.array_equal(q, layer.w.w2_q[int(e)].cpu().numpy()), f"W2 codes of expert {e}"
        w[2].append(q); w[3].append(s)
    w = [np.stack(a) for a in w]
    xq, xs = oracle.quant_1x128(bf16_bits(x[torch.as_tensor(tokens, device=DEV)]))
    rows_q = np.repeat(xq, k, axis=0)
    rows_s = np.repeat(xs, k, axis=0)
    row_e = np.array([remap[int(e)] for e in ids.reshape(-1)], np.int32)
    _, _, _, out = oracle.expert_ffn(rows_q, rows_s, row_e, *w)
    sl2 = np.arange(len(tokens) * k, dtype=np.int32)
    return oracle.combine(out, sl2, gates_ref)


def test_large_full_size(L, oracle, parity_report):
    cfg = S.CONFIGS["large"]
    layer = _layer(cfg)
    x = S.make_x(cfg, DEV)
    cap = torch.empty((cfg.k, cfg.T), dtype=torch.int32, device=DEV)
    y = layer.forward(x, capture_kT=cap)
    torch.cuda.synchronize()
    assert L.check_status(layer.dev_status) == 0
    ids_gpu = layer.ids.cpu().numpy()
    assert np.array_equal(cap.cpu().numpy(), ids_gpu.T)
    # routing of every token by the oracle (15 G fmas on the host cores)
    xb = bf16_bits(x)
    lg_all = oracle.router_logits(xb, bf16_bits(layer.w.w_router))
    ids_all = oracle.topk(lg_all, cfg.k)
    np.testing.assert_array_equal(ids_gpu, ids_all)
    tokens = np.arange(cfg.T)
    ids_ref = ids_all[tokens]
    g_ref = oracle.gates(lg_all[tokens], ids_ref, cfg.score_fn, cfg.renorm, cfg.route_scale)
    np.testing.assert_allclose(layer.gates[torch.as_tensor(tokens, device=DEV)].cpu().numpy(), g_ref, rtol=1e-5)
    counts, offsets, s2s, sl2, _ = oracle.dispatch(ids_all, cfg.E)
    np.testing.assert_array_equal(layer.offsets.cpu().numpy(), offsets)
    np.testing.assert_array_equal(layer.sl2.cpu().numpy(), sl2)
    A = cfg.T * cfg.k
    np.testing.assert_array_equal(layer.s2s[:A].cpu().numpy(), s2s)
    xq, xs = oracle.quant_1x128(xb)
    np.testing.assert_array_equal(layer.xq.cpu().numpy(), xq)
    np.testing.assert_array_equal(layer.xs.cpu().numpy(), xs)
    np.testing.assert_array_equal(layer.xq_sorted.cpu().numpy(), oracle.gather_rows(xq, s2s, A, cfg.k))
    y_ref = _oracle_tokens(oracle, cfg, layer, tokens, ids_ref, g_ref, x)
    err = parity_report("large layer y, all tokens", bf16_to_f64(bf16_bits(y)), bf16_to_f64(y_ref))
    assert err.max() <= TOL, err.max()


def test_long_dispatch_full_size(L, oracle):
    cfg = S.CONFIGS["long_dispatch"]
    payload = S.make_replay_payload(cfg, DEV)[0]
    gates = S.make_dirichlet_gates(cfg, DEV)
    x = S.make_x(cfg, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids, _ = L.moe_route_replay(payload, cfg.E, dev_status=st)
    counts, offsets, s2s, sl2, rows, _ = L.moe_dispatch(ids, cfg.E, rows=x, dev_status=st)
    y = L.moe_combine(rows, sl2, gates)
    torch.cuda.synchronize()
    assert L.check_status(st) == 0
    rid, valid, bad = oracle.replay(payload.cpu().numpy(), cfg.E)
    assert bad == 0
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    rc, ro, rs2s, rsl2, _ = oracle.dispatch(rid, cfg.E)
    np.testing.assert_array_equal(counts.cpu().numpy(), rc)
    np.testing.assert_array_equal(offsets.cpu().numpy(), ro)
    np.testing.assert_array_equal(s2s.cpu().numpy(), rs2s)
    np.testing.assert_array_equal(sl2.cpu().numpy(), rsl2)
    # every dispatched row is its token's row (checked on the device)
    tok = torch.as_tensor(rs2s // cfg.k, device=DEV, dtype=torch.int64)
    for c in range(0, tok.numel(), 1 << 18):
        assert torch.equal(rows[c:c + (1 << 18)].view(torch.int16), x[tok[c:c + (1 << 18)]].view(torch.int16))
    assert torch.equal(y.view(torch.int16), x.view(torch.int16))


def test_multilayer_replay_all_layers(L, oracle, parity_report):
    cfg = S.CONFIGS["multilayer_replay"]
    payload = S.make_replay_payload(cfg, DEV)           # [8, 8, 16384]
    assert payload.shape == (8, cfg.k, cfg.T)
    for l in range(cfg.layers):
        layer = _layer(cfg, layer_idx=l)
        x = S.make_x(cfg, DEV, layer=l)
        slab = payload[l]
        y = layer.forward(x, replay_kT=slab)
        torch.cuda.synchronize()
        assert L.check_status(layer.dev_status) == 0
        rid, valid, bad = oracle.replay(slab.cpu().numpy(), cfg.E)
        assert bad == 0
        np.testing.assert_array_equal(layer.ids.cpu().numpy(), rid)
        counts, offsets, s2s, sl2, _ = oracle.dispatch(rid, cfg.E)
        np.testing.assert_array_equal(layer.counts.cpu().numpy(), counts)
        np.testing.assert_array_equal(layer.sl2.cpu().numpy(), sl2)
        assert (counts == 0).sum() == cfg.n_cold
        hot = np.argsort(counts)[::-1][: cfg.n_hot]
        rng = np.random.default_rng(l)
        tokens = [int(np.nonzero((rid == h).any(axis=1))[0][0]) for h in hot]
        tokens = np.unique(np.concatenate([tokens, rng.choice(cfg.T, 2048 - len(tokens), replace=False)]))
        xb = bf16_bits(x[torch.as_tensor(tokens, device=DEV)])
        lg = oracle.router_logits(xb, bf16_bits(layer.w.w_router))
        g_ref = oracle.gates(lg, rid[tokens], cfg.score_fn, cfg.renorm, cfg.route_scale)
        np.testing.assert_allclose(layer.gates[torch.as_tensor(tokens, device=DEV)].cpu().numpy(), g_ref,
                                   rtol=1e-5)
        y_ref = _oracle_tokens(oracle, cfg, layer, tokens, rid[tokens], g_ref, x, layer_idx=l)
        err = parity_report(f"replay layer {l} y, sampled tokens",
                            bf16_to_f64(bf16_bits(y[torch.as_tensor(tokens, device=DEV)])), bf16_to_f64(y_ref))
        assert err.max() <= TOL, err.max()
        del layer
        torch.cuda.empty_cache()


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (333, 8, 2), (40, 1, 1), (129, 16, 16)])
def test_layer_ragged_and_degenerate(L, oracle, parity_report, T, E, k):
    """A single token, a ragged token count, a single expert (k = 1), and
    k = E (every token to every expert)."""
    from block_scaled_fp8_router_gb300.layer import MoELayerFP8, MoEWeightsFP8, quantize_weights
    cfg = S.CONFIGS["tiny"].with_(T=T, E=E, k=k)
    x = S.make_x(cfg, DEV)
    wr = S.make_router_w(cfg, DEV)
    w13, w2 = S.make_w13(cfg, DEV), S.make_w2(cfg, DEV)
    layer = MoELayerFP8(MoEWeightsFP8(wr, *quantize_weights(w13, w2)), T, k, cfg.score_fn)
    y = layer.forward(x)
    torch.cuda.synchronize()
    xb = bf16_bits(x)
    lg = oracle.router_logits(xb, bf16_bits(wr))
    ids = oracle.topk(lg, k)
    np.testing.assert_array_equal(layer.ids.cpu().numpy(), ids)
    g = oracle.gates(lg, ids, cfg.score_fn, 1, 1.0)
    y_ref = _oracle_tokens(oracle, cfg, layer, np.arange(T), ids, g, x)
    err = parity_report(f"y T={T} E={E} k={k}", bf16_to_f64(bf16_bits(y)), bf16_to_f64(y_ref))
    assert err.max() <= TOL, err.max()
