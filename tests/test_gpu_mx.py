"""GPU parity of the power-of-two (UE8M0) variant against the CPU oracle:
the quantiser bit for bit (codes and exponent bytes), and the grouped FFN on
the hardware block-scaled MMA (tcgen05.mma.kind::mxf8f6f4.block_scale)
within the layer's 2e-2 row-relative bar (the tensor core accumulates the
whole K extent in fp32 where the oracle promotes exact 128-deep block
products one by one; act codes may flip where act / scale sits on a
rounding midpoint)."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_router_gb300 import synthetic as S
from tests.helpers import bf16_bits, bf16_to_f64, e4m3_to_f64, row_rel_err

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
TOL = 2e-2


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from block_scaled_fp8_router_gb300 import moe_r3
    return moe_r3


def _edge_rows(rows, cols, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn(rows, cols, generator=g, device=DEV)
    x = (x * torch.exp2(torch.randint(-30, 30, (rows, 1), generator=g, device=DEV).float())).to(torch.bfloat16)
    x[0, :128] = 0.0
    x[1, 128:256] = -0.0
    x[2, :128] = 1e-40
    x[3, :128] = 448.0
    x[3, 5] = -448.0 * (1 + 2.0 ** -7)
    x[4, :128] = 3.0e38
    x[5, :128] = 2.0 ** -130
    return x


@pytest.mark.parametrize("rows,cols", [(6, 256), (1000, 7168 // 2), (37, 2048)])
def test_quant_ue8m0_1x128_bit_exact(L, oracle, rows, cols):
    x = _edge_rows(max(rows, 6), cols, rows + cols)
    q, e = L.fp8_block_quant_ue8m0(x, 1)
    rq, re_ = oracle.quant_ue8m0(bf16_bits(x), 1)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(e.cpu().numpy(), re_)


def test_quant_ue8m0_128x128_bit_exact(L, oracle):
    cfg = S.CONFIGS["tiny"]
    w = torch.cat([S.make_w13_expert(cfg, 0, DEV), S.make_w13_expert(cfg, 1, DEV) * 300.0]).contiguous()
    w[:128, :128] = 0
    q, e = L.fp8_block_quant_ue8m0(w, 128)
    rq, re_ = oracle.quant_ue8m0(bf16_bits(w), 128)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(e.cpu().numpy(), re_)


def _quant_weights_mx(L, w13, w2):
    E, twoF, d = w13.shape
    F = w2.shape[2]
    q13, e13 = L.fp8_block_quant_ue8m0(w13.reshape(E * twoF, d), 128)
    q2, e2 = L.fp8_block_quant_ue8m0(w2.reshape(E * d, F), 128)
    return (q13.view(E, twoF, d), e13.view(E, twoF // 128, d // 128), q2.view(E, d, F), e2.view(E, d // 128, F // 128))


def _run_mx(L, counts, d, F, k=1, seed=0):
    """Rows of expert e are tokens in a seeded order (sorted_to_slot a
    permutation of T*k slots, k = 1 or more) so the token-major exponent
    lookup is exercised."""
    E = len(counts)
    cfg = S.CONFIGS["tiny"].with_(d=d, F=F, E=E, w_std=0.02)
    w13 = torch.stack([S.make_w13_expert(cfg, e, DEV, seed) for e in range(E)])
    w2 = torch.stack([S.make_w2_expert(cfg, e, DEV, seed) for e in range(E)])
    wq = _quant_weights_mx(L, w13, w2)
    A = int(sum(counts))
    T = (A + k - 1) // k
    g = torch.Generator(device=DEV).manual_seed(seed + 1)
    x = torch.randn((T, d), generator=g, device=DEV).to(torch.bfloat16)
    xq, xe = L.fp8_block_quant_ue8m0(x, 1)
    s2s = torch.randperm(T * k, generator=g, device=DEV)[:A].to(torch.int32)
    xq_sorted = xq[(s2s // k).long()].contiguous() if A else torch.zeros((1, d), dtype=torch.uint8, device=DEV)
    mr = max(A, 1)
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device=DEV)
    out = torch.full((mr, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(L.moe_grouped_ffn_mx_workspace_size(mr, d, F), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    s2s_arg = s2s if A else torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_grouped_ffn_mx(xq_sorted, xe, s2s_arg, k, offsets, *wq, out_sorted=out, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    return dict(x=x, s2s=s2s, k=k, w13=w13, w2=w2, out=out, ws=ws, st=L.check_status(st), A=A, mr=mr,
                counts=counts)


def _oracle_mx(oracle, r):
    counts = r["counts"]
    A = r["A"]
    row_e = np.repeat(np.arange(len(counts), dtype=np.int32), counts)
    tok = (r["s2s"].cpu().numpy() // r["k"]).astype(np.int64)
    xq, xe = oracle.quant_ue8m0(bf16_bits(r["x"]), 1)
    f = oracle.ue8m0_value
    w = []
    for e in range(len(counts)):
        w.append((oracle.quant_ue8m0(bf16_bits(r["w13"][e]), 128), oracle.quant_ue8m0(bf16_bits(r["w2"][e]), 128)))
    w13q = np.stack([a[0][0] for a in w]); w13s = np.stack([f(a[0][1]) for a in w])
    w2q = np.stack([a[1][0] for a in w]); w2s = np.stack([f(a[1][1]) for a in w])
    return oracle.expert_ffn(xq[tok], f(xe[tok]), row_e, w13q, w13s, w2q, w2s, ue8m0=True)


@pytest.mark.parametrize("counts,d,F,k", [
    ([128], 128, 128, 1),
    ([1, 127, 128, 129, 300, 0, 5], 256, 256, 2),
    ([0, 0, 200, 0], 256, 384, 1),
    ([260, 3, 0, 64], 384, 256, 4),          # d % 256 == 128: GEMM2 N tail
])
def test_grouped_ffn_mx_against_oracle(L, oracle, counts, d, F, k):
    r = _run_mx(L, counts, d, F, k, seed=len(counts) + d)
    assert r["st"] == 0
    A = r["A"]
    act_f, act_q, act_s, out = _oracle_mx(oracle, r)
    ws = r["ws"].cpu().numpy()
    g_actq = ws[: A * F].reshape(A, F)
    off = (r["mr"] * F + 255) // 256 * 256
    g_acte = ws[off: off + A * (F // 128)].reshape(A, F // 128)
    g_act = e4m3_to_f64(g_actq) * np.repeat(np.ldexp(1.0, g_acte.astype(np.int64) - 127), 128, axis=1)
    ref_act = e4m3_to_f64(act_q) * np.repeat(act_s.astype(np.float64), 128, axis=1)
    assert row_rel_err(g_act, ref_act).max() <= TOL
    flips = (g_actq != act_q).mean()
    assert flips < 1e-2, flips
    err = row_rel_err(bf16_to_f64(bf16_bits(r["out"][:A])), bf16_to_f64(out))
    assert err.max() <= TOL, err.max()
    print(f"counts={counts} d={d} F={F}: max row rel err {err.max():.2e}, act code flips {flips:.1e}")


def test_grouped_ffn_mx_all_empty(L):
    r = _run_mx(L, [0, 0, 0], 256, 256)
    assert r["st"] == 0


def _mx_layer(cfg, seed=0):
    from block_scaled_fp8_router_gb300.layer import MoELayerFP8, MoEWeightsFP8, quantize_weights
    E, d, F = cfg.E, cfg.d, cfg.F
    w = MoEWeightsFP8(S.make_router_w(cfg, DEV, seed),
                      torch.empty((E, 2 * F, d), dtype=torch.uint8, device=DEV),
                      torch.empty((E, 2 * F // 128, d // 128), dtype=torch.uint8, device=DEV),
                      torch.empty((E, d, F), dtype=torch.uint8, device=DEV),
                      torch.empty((E, d // 128, F // 128), dtype=torch.uint8, device=DEV))
    for e0 in range(0, E, 16):
        n = min(16, E - e0)
        w13 = torch.stack([S.make_w13_expert(cfg, e, DEV, seed) for e in range(e0, e0 + n)])
        w2 = torch.stack([S.make_w2_expert(cfg, e, DEV, seed) for e in range(e0, e0 + n)])
        quantize_weights(w13, w2, out=w, e0=e0)
    return MoELayerFP8(w, cfg.T, cfg.k, cfg.score_fn, cfg.renorm, cfg.route_scale)


def _oracle_mx_tokens(oracle, cfg, layer, tokens, ids, gates_ref, x, seed=0):
    """Oracle output of the sampled tokens with power-of-two scales (every
    expert row they use), the experts' exponent bytes checked against the GPU."""
    k = cfg.k
    used = np.unique(ids)
    remap = {int(e): i for i, e in enumerate(used)}
    f = oracle.ue8m0_value
    w = [[], [], [], []]
    for e in used:
        q, ee = oracle.quant_ue8m0(bf16_bits(S.make_w13_expert(cfg, int(e), DEV, seed)), 128)
        assert np.array_equal(q, layer.w.w13_q[int(e)].cpu().numpy())
        assert np.array_equal(ee, layer.w.w13_s[int(e)].cpu().numpy())
        w[0].append(q); w[1].append(f(ee))
        q, ee = oracle.quant_ue8m0(bf16_bits(S.make_w2_expert(cfg, int(e), DEV, seed)), 128)
        assert np.array_equal(ee, layer.w.w2_s[int(e)].cpu().numpy())
        w[2].append(q); w[3].append(f(ee))
    w = [np.stack(a) for a in w]
    xq, xe = oracle.quant_ue8m0(bf16_bits(x[torch.as_tensor(tokens, device=DEV)]), 1)
    row_e = np.array([remap[int(e)] for e in ids.reshape(-1)], np.int32)
    _, _, _, out = oracle.expert_ffn(np.repeat(xq, k, axis=0), np.repeat(f(xe), k, axis=0), row_e, *w, ue8m0=True)
    return oracle.combine(out, np.arange(len(tokens) * k, dtype=np.int32), gates_ref)


@pytest.mark.parametrize("name,T", [("tiny", None), ("replay", 600)])
def test_mx_layer_against_oracle(L, oracle, parity_report, name, T):
    cfg = S.CONFIGS[name]
    if T:
        cfg = cfg.with_(T=T)
    layer = _mx_layer(cfg)
    x = S.make_x(cfg, DEV)
    replay = S.make_replay_payload(cfg.with_(layers=1), DEV)[0] if cfg.mode == "replay" else None
    y = layer.forward(x, replay_kT=replay)
    torch.cuda.synchronize()
    assert L.check_status(layer.dev_status) == 0
    xb = bf16_bits(x)
    lg = oracle.router_logits(xb, bf16_bits(layer.w.w_router))
    ids = oracle.topk(lg, cfg.k) if replay is None else oracle.replay(replay.cpu().numpy(), cfg.E)[0]
    np.testing.assert_array_equal(layer.ids.cpu().numpy(), ids)
    q, e = oracle.quant_ue8m0(xb, 1)
    np.testing.assert_array_equal(layer.xq.cpu().numpy(), q)
    np.testing.assert_array_equal(layer.xs.cpu().numpy(), e)
    g = oracle.gates(lg, ids, cfg.score_fn, cfg.renorm, cfg.route_scale)
    tokens = np.arange(cfg.T)
    y_ref = _oracle_mx_tokens(oracle, cfg, layer, tokens, ids, g, x)
    err = parity_report("power-of-two layer y", bf16_to_f64(bf16_bits(y)), bf16_to_f64(y_ref))
    assert err.max() <= TOL, err.max()
    print(f"mx layer {name}: max row rel err {err.max():.2e}")


def test_mx_layer_full_size_sampled(L, oracle, parity_report):
    """The 8192-token large layer with power-of-two scales: ids, codes and
    exponents of x in full, and the output of 64 sampled tokens."""
    cfg = S.CONFIGS["large"]
    layer = _mx_layer(cfg)
    x = S.make_x(cfg, DEV)
    y = layer.forward(x)
    torch.cuda.synchronize()
    assert L.check_status(layer.dev_status) == 0
    xb = bf16_bits(x)
    q, e = oracle.quant_ue8m0(xb, 1)
    np.testing.assert_array_equal(layer.xq.cpu().numpy(), q)
    np.testing.assert_array_equal(layer.xs.cpu().numpy(), e)
    rng = np.random.default_rng(1)
    tokens = np.sort(np.concatenate([[0, cfg.T - 1], rng.choice(np.arange(1, cfg.T - 1), 62, replace=False)]))
    lg = oracle.router_logits(xb[tokens], bf16_bits(layer.w.w_router))
    ids = oracle.topk(lg, cfg.k)
    np.testing.assert_array_equal(layer.ids[torch.as_tensor(tokens, device=DEV)].cpu().numpy(), ids)
    g = oracle.gates(lg, ids, cfg.score_fn, cfg.renorm, cfg.route_scale)
    y_ref = _oracle_mx_tokens(oracle, cfg, layer, tokens, ids, g, x)
    err = parity_report("power-of-two large y, sampled", bf16_to_f64(bf16_bits(y[torch.as_tensor(tokens, device=DEV)])),
                        bf16_to_f64(y_ref))
    assert err.max() <= TOL, err.max()
    print(f"mx large: {len(tokens)} sampled tokens, max row rel err {err.max():.2e}")
