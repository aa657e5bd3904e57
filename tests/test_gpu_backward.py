"""GPU parity of the expert path's backward under replay against the CPU
oracle, through the C ABI: combine backward (quantised gradient rows and
scales bit-exact, gate gradients to fp32 accumulation), the weight
transpose and the dispatch backward bit-exact, the saved GEMM1
pre-activations and both dgrad GEMMs within the layer's 2e-2 row bar, the
SwiGLU backward within rounding (code flips < 1%), and the composed
backward of the layer against the oracle's chain, every token on the tiny
and replay workloads and a token sample of the 8192-token layer."""
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


def _layer(cfg, T=None):
    from block_scaled_fp8_router_gb300.layer import MoELayerFP8, MoEWeightsFP8, quantize_weights
    wr = S.make_router_w(cfg, DEV)
    w13, w2 = S.make_w13(cfg, DEV), S.make_w2(cfg, DEV)
    w = MoEWeightsFP8(wr, *quantize_weights(w13, w2))
    return MoELayerFP8(w, T or cfg.T, cfg.k, cfg.score_fn, cfg.renorm, cfg.route_scale)


def _deq_rows(q, s):
    return e4m3_to_f64(q) * np.repeat(s.astype(np.float64), 128, axis=1)


@pytest.mark.parametrize("T,k,d", [(37, 3, 256), (300, 8, 384), (5, 1, 128), (700, 8, 7168), (9, 2, 16512)])
def test_combine_backward_against_oracle(L, oracle, T, k, d):
    """Rows staged by bulk copies (d <= 8192; T above the persistent grid at
    d = 7168, so CTAs take several tokens and wrap the stage ring) and the
    register path past that (d = 16512)."""
    g = torch.Generator(device=DEV).manual_seed(T + d)
    A = T * k
    sl2 = torch.randperm(A, generator=g, device=DEV).to(torch.int32)
    sl2[::7] = -1
    out = torch.randn((A, d), generator=g, device=DEV).to(torch.bfloat16)
    dy = torch.randn((T, d), generator=g, device=DEV).to(torch.bfloat16)
    gates = torch.rand((T, k), generator=g, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dq, ds, dg = L.moe_combine_backward(dy, gates, out, sl2, dev_status=st)
    assert int(st.item()) == 0
    rf, rq, rs, rg = oracle.combine_backward(bf16_bits(dy), gates.cpu().numpy(), bf16_bits(out), sl2.cpu().numpy())
    s = sl2.cpu().numpy()
    routed = s[s >= 0]
    np.testing.assert_array_equal(dq.cpu().numpy()[routed], rq[routed])
    np.testing.assert_array_equal(ds.cpu().numpy()[routed], rs[routed])
    idx = np.where(s >= 0, s, 0)
    mag = (np.abs(bf16_to_f64(bf16_bits(dy)))[:, None, :] *
           np.abs(bf16_to_f64(bf16_bits(out)))[idx].reshape(T, k, d)).sum(2)
    assert np.all(np.abs(dg.cpu().numpy() - rg) <= mag * 1e-6 + 1e-30)
    assert np.all(dg.cpu().numpy().reshape(-1)[s < 0] == 0)


def test_weight_transpose_bit_exact(L, oracle):
    cfg = S.CONFIGS["tiny"]
    from block_scaled_fp8_router_gb300.layer import quantize_weights
    w13, w2 = S.make_w13(cfg, DEV), S.make_w2(cfg, DEV)
    w13q, w13s, w2q, w2s = quantize_weights(w13, w2)
    for q, s_ in ((w13q, w13s), (w2q, w2s)):
        qt, st = L.fp8_weight_transpose(q, s_)
        rq, rs = oracle.weight_transpose(q.cpu().numpy(), s_.cpu().numpy())
        np.testing.assert_array_equal(qt.cpu().numpy(), rq)
        np.testing.assert_array_equal(st.cpu().numpy(), rs)


def test_dispatch_backward_bit_exact(L, oracle):
    g = torch.Generator(device=DEV).manual_seed(3)
    T, k, d = 211, 8, 384
    A = T * k
    sl2 = torch.randperm(A, generator=g, device=DEV).to(torch.int32)
    sl2[::11] = -1
    rows = torch.randn((A, d), generator=g, device=DEV).to(torch.bfloat16)
    dx = L.moe_dispatch_backward(rows, sl2, T, k)
    ref = oracle.dispatch_backward(bf16_bits(rows), sl2.cpu().numpy(), T, k)
    np.testing.assert_array_equal(bf16_bits(dx), ref)


def _oracle_backward(oracle, layer, x, dy, T, k):
    """The oracle's chain on the layer's own routing: every sorted row."""
    E, d, F = layer.w.E, layer.w.d, layer.w.F
    A = T * k
    xq, xs = oracle.quant_1x128(bf16_bits(x))
    s2s = layer.s2s[:A].cpu().numpy()
    sl2 = layer.sl2[:A].cpu().numpy()
    counts = layer.counts.cpu().numpy()
    row_e = np.repeat(np.arange(E, dtype=np.int32), counts)
    rows_q = oracle.gather_rows(xq, s2s, A, k)
    rows_s = oracle.gather_rows(xs, s2s, A, k)
    w13q, w13s = layer.w.w13_q.cpu().numpy(), layer.w.w13_s.cpu().numpy()
    w2q, w2s = layer.w.w2_q.cpu().numpy(), layer.w.w2_s.cpu().numpy()
    h = oracle.expert_ffn_preact(rows_q, rows_s, row_e, w13q, w13s)
    _, _, _, out = oracle.expert_ffn(rows_q, rows_s, row_e, w13q, w13s, w2q, w2s)
    _, dq, ds, dg = oracle.combine_backward(bf16_bits(dy), layer.gates[:T].cpu().numpy(), out, sl2)
    w2tq, w2ts = oracle.weight_transpose(w2q, w2s)
    w13tq, w13ts = oracle.weight_transpose(w13q, w13s)
    d_act = oracle.grouped_gemm(dq, ds, row_e, w2tq, w2ts)
    _, dhq, dhs = oracle.swiglu_backward(d_act, h)
    dxs = oracle.grouped_gemm(dhq, dhs, row_e, w13tq, w13ts)
    dx = oracle.dispatch_backward(dxs, sl2, T, k)
    return dict(h=h, d_out_q=dq, d_out_s=ds, d_gates=dg, d_act=d_act, dh_q=dhq, dh_s=dhs, dx_sorted=dxs, dx=dx)


@pytest.mark.parametrize("name,T", [("tiny", None), ("replay", 500)])
def test_layer_backward_against_oracle(L, oracle, parity_report, name, T):
    cfg = S.CONFIGS[name]
    if T:
        cfg = cfg.with_(T=T)
    layer = _layer(cfg)
    x = S.make_x(cfg, DEV)
    replay = S.make_replay_payload(cfg.with_(layers=1), DEV)[0] if cfg.mode == "replay" else None
    y_ref_form = layer.forward(x, replay_kT=replay).clone()
    y = layer.forward(x, replay_kT=replay, train=True)
    assert torch.equal(y.view(torch.int16), y_ref_form.view(torch.int16))       # saving h changes nothing
    g = torch.Generator(device=DEV).manual_seed(5)
    dy = torch.randn((cfg.T, cfg.d), generator=g, device=DEV).to(torch.bfloat16)
    dx, d_gates = layer.backward(dy)
    torch.cuda.synchronize()
    assert L.check_status(layer.dev_status) == 0
    A = cfg.T * cfg.k
    r = _oracle_backward(oracle, layer, x, dy, cfg.T, cfg.k)
    b = layer._bw
    assert row_rel_err(layer.h[:A].cpu().numpy().astype(np.float64), r["h"].astype(np.float64)).max() <= 1e-5
    np.testing.assert_array_equal(b["d_out_q"][:A].cpu().numpy(), r["d_out_q"])  # g * dy only: same gates, same codes
    e_act = row_rel_err(bf16_to_f64(bf16_bits(b["d_act"][:A])), bf16_to_f64(r["d_act"]))
    assert e_act.max() <= TOL, e_act.max()
    g_dh = _deq_rows(b["dh_q"][:A].cpu().numpy(), b["dh_s"][:A].cpu().numpy())
    r_dh = _deq_rows(r["dh_q"], r["dh_s"])
    assert row_rel_err(g_dh, r_dh).max() <= TOL
    assert (b["dh_q"][:A].cpu().numpy() != r["dh_q"]).mean() < 1e-2
    e_dxs = row_rel_err(bf16_to_f64(bf16_bits(b["dx_sorted"][:A])), bf16_to_f64(r["dx_sorted"]))
    assert e_dxs.max() <= TOL, e_dxs.max()
    e_dx = parity_report("backward dx", bf16_to_f64(bf16_bits(dx)), bf16_to_f64(r["dx"]))
    assert e_dx.max() <= TOL, e_dx.max()
    mag = np.abs(r["d_gates"]).max()
    assert np.abs(d_gates.cpu().numpy() - r["d_gates"]).max() <= 2e-2 * mag
    print(f"{name}: backward max row rel err d_act {e_act.max():.2e} dx_sorted {e_dxs.max():.2e} dx {e_dx.max():.2e}")


def test_backward_full_size_sampled(L, oracle):
    """The 8192-token large layer (d=7168, E=256, top-8, F=2048): forward with
    the pre-activations kept, backward of the expert path, and the oracle's
    chain on 64 sampled tokens (every row is independent given its routing)."""
    cfg = S.CONFIGS["large"]
    from tests.test_gpu_fullsize import _layer as big_layer
    layer = big_layer(cfg)
    x = S.make_x(cfg, DEV)
    layer.forward(x, train=True)
    g = torch.Generator(device=DEV).manual_seed(9)
    dy = torch.randn((cfg.T, cfg.d), generator=g, device=DEV).to(torch.bfloat16)
    dx, d_gates = layer.backward(dy)
    torch.cuda.synchronize()
    assert L.check_status(layer.dev_status) == 0
    rng = np.random.default_rng(2)
    tokens = np.sort(np.concatenate([[0, cfg.T - 1], rng.choice(np.arange(1, cfg.T - 1), 62, replace=False)]))
    k = cfg.k
    n = len(tokens)
    tt = torch.as_tensor(tokens, device=DEV)
    ids = layer.ids[tt].cpu().numpy()
    used = np.unique(ids)
    remap = {int(e): i for i, e in enumerate(used)}
    row_e = np.array([remap[int(e)] for e in ids.reshape(-1)], np.int32)
    w13q = layer.w.w13_q[torch.as_tensor(used, device=DEV)].cpu().numpy()
    w13s = layer.w.w13_s[torch.as_tensor(used, device=DEV)].cpu().numpy()
    w2q = layer.w.w2_q[torch.as_tensor(used, device=DEV)].cpu().numpy()
    w2s = layer.w.w2_s[torch.as_tensor(used, device=DEV)].cpu().numpy()
    xq, xs = oracle.quant_1x128(bf16_bits(x[tt]))
    rq, rs = np.repeat(xq, k, axis=0), np.repeat(xs, k, axis=0)
    h = oracle.expert_ffn_preact(rq, rs, row_e, w13q, w13s)
    _, _, _, out = oracle.expert_ffn(rq, rs, row_e, w13q, w13s, w2q, w2s)
    loc = np.arange(n * k, dtype=np.int32)
    _, dq, ds, dg = oracle.combine_backward(bf16_bits(dy[tt]), layer.gates[tt].cpu().numpy(), out, loc)
    w2tq, w2ts = oracle.weight_transpose(w2q, w2s)
    w13tq, w13ts = oracle.weight_transpose(w13q, w13s)
    d_act = oracle.grouped_gemm(dq, ds, row_e, w2tq, w2ts)
    _, dhq, dhs = oracle.swiglu_backward(d_act, h)
    dxs = oracle.grouped_gemm(dhq, dhs, row_e, w13tq, w13ts)
    dx_ref = oracle.dispatch_backward(dxs, loc, n, k)
    # the GPU's quantised gradient rows of the sampled slots are bit-exact
    sl2 = layer.sl2.cpu().numpy().reshape(cfg.T, k)[tokens].reshape(-1)
    np.testing.assert_array_equal(layer._bw["d_out_q"][torch.as_tensor(sl2, device=DEV)].cpu().numpy(), dq)
    err = row_rel_err(bf16_to_f64(bf16_bits(dx[tt])), bf16_to_f64(dx_ref))
    assert err.max() <= TOL, err.max()
    mag = np.abs(dg).max()
    assert np.abs(d_gates[tt].cpu().numpy() - dg).max() <= 2e-2 * mag
    print(f"large backward: {n} sampled tokens, max row rel err dx {err.max():.2e}")


@pytest.mark.parametrize("name,T", [("tiny", None), ("replay", 500)])
def test_weight_gradients_against_oracle(L, oracle, name, T):
    """dW2 = d_out^T act and dW13 = dh^T x per expert from 128 x 1 operands:
    the d_out and x operands bit-exact (same values on both sides), act and
    dh within rounding (code flips < 1%), and both gradients within 2e-2 of
    each expert matrix's largest entry."""
    cfg = S.CONFIGS[name]
    if T:
        cfg = cfg.with_(T=T)
    layer = _layer(cfg)
    x = S.make_x(cfg, DEV)
    replay = S.make_replay_payload(cfg.with_(layers=1), DEV)[0] if cfg.mode == "replay" else None
    layer.forward(x, replay_kT=replay, train=True)
    g = torch.Generator(device=DEV).manual_seed(8)
    dy = torch.randn((cfg.T, cfg.d), generator=g, device=DEV).to(torch.bfloat16)
    dx, d_gates, dW13, dW2 = layer.backward(dy, weight_grads=True)
    torch.cuda.synchronize()
    assert L.check_status(layer.dev_status) == 0
    E, d, F, k, Tn = cfg.E, cfg.d, cfg.F, cfg.k, cfg.T
    A = Tn * k
    offsets = layer.offsets.cpu().numpy()
    s2s = layer.s2s[:A].cpu().numpy()
    sl2 = layer.sl2[:A].cpu().numpy()
    counts = layer.counts.cpu().numpy()
    row_e = np.repeat(np.arange(E, dtype=np.int32), counts)
    xq, xs = oracle.quant_1x128(bf16_bits(x))
    rq, rs = oracle.gather_rows(xq, s2s, A, k), oracle.gather_rows(xs, s2s, A, k)
    w13q, w13s = layer.w.w13_q.cpu().numpy(), layer.w.w13_s.cpu().numpy()
    w2q, w2s = layer.w.w2_q.cpu().numpy(), layer.w.w2_s.cpu().numpy()
    h = oracle.expert_ffn_preact(rq, rs, row_e, w13q, w13s)
    act_f, _, _, out = oracle.expert_ffn(rq, rs, row_e, w13q, w13s, w2q, w2s)
    d_out_f, dq, ds, _ = oracle.combine_backward(bf16_bits(dy), layer.gates[:Tn].cpu().numpy(), out, sl2)
    w2tq, w2ts = oracle.weight_transpose(w2q, w2s)
    d_act = oracle.grouped_gemm(dq, ds, row_e, w2tq, w2ts)
    dh_f, _, _ = oracle.swiglu_backward(d_act, h)
    x_rows = bf16_to_f64(bf16_bits(x)).astype(np.float32)[s2s // k]
    # operands: d_out and x bit-exact against the oracle's 128 x 1 quantisation
    pad = L.moe_wgrad_pad_offsets(layer.offsets)
    ld = L.wgrad_ld(A, E)
    gq, gs = L.moe_wgrad_quant(L.WGRAD_SRC_GDY, layer.offsets, pad, d, ld, False, dy=dy, gates=layer.gates[:Tn],
                               sorted_to_slot=layer.s2s[:A], k=k)
    gq2, gs2 = L.moe_wgrad_quant(L.WGRAD_SRC_GDY, layer.offsets, pad, d, ld, True, dy=dy, gates=layer.gates[:Tn],
                                 sorted_to_slot=layer.s2s[:A], k=k)
    oq, os_, opad = oracle.quant_128x1(d_out_f, offsets)
    np.testing.assert_array_equal(pad.cpu().numpy(), opad)
    P = int(opad[-1])
    np.testing.assert_array_equal(gq.cpu().numpy()[:, :P], oq)
    np.testing.assert_array_equal(gs.cpu().numpy()[:, :P // 128], os_)
    np.testing.assert_array_equal(gq2.cpu().numpy()[:, :P], oq)                  # both scale layouts
    np.testing.assert_array_equal(gs2.cpu().numpy()[:P // 128].T, os_)
    xq2, xs2 = L.moe_wgrad_quant(L.WGRAD_SRC_X, layer.offsets, pad, d, ld, True, x=x, sorted_to_slot=layer.s2s[:A], k=k)
    oxq, oxs, _ = oracle.quant_128x1(x_rows, offsets)
    np.testing.assert_array_equal(xq2.cpu().numpy()[:, :P], oxq)
    np.testing.assert_array_equal(xs2.cpu().numpy()[:P // 128].T, oxs)
    aq2, _ = L.moe_wgrad_quant(L.WGRAD_SRC_ACT, layer.offsets, pad, F, ld, True, h=layer.h, F=F)
    oaq, oas, _ = oracle.quant_128x1(act_f, offsets)
    assert (aq2.cpu().numpy()[:, :P] != oaq).mean() < 1e-2
    # the gradients
    ohq, ohs, _ = oracle.quant_128x1(dh_f, offsets)
    dW2_ref = oracle.wgrad(oq, os_, oaq, oas, opad)
    dW13_ref = oracle.wgrad(ohq, ohs, oxq, oxs, opad)
    for got, ref, nm in ((dW2.cpu().numpy(), dW2_ref, "dW2"), (dW13.cpu().numpy(), dW13_ref, "dW13")):
        for e in range(E):
            if counts[e] == 0:
                assert np.all(got[e] == 0)
                continue
            err = np.abs(got[e] - ref[e]).max() / max(np.abs(ref[e]).max(), 1e-30)
            assert err <= TOL, (nm, e, err)
    print(f"{name}: weight gradients within {TOL} of each expert's largest entry")


def test_weight_gradients_full_size_two_experts(L, oracle):
    """The 8192-token large layer: dW2 and dW13 of two experts (the most and
    the least loaded) against the oracle's chain on those experts' rows
    (every expert's gradient depends only on its own rows)."""
    cfg = S.CONFIGS["large"]
    from tests.test_gpu_fullsize import _layer as big_layer
    layer = big_layer(cfg)
    x = S.make_x(cfg, DEV)
    layer.forward(x, train=True)
    g = torch.Generator(device=DEV).manual_seed(12)
    dy = torch.randn((cfg.T, cfg.d), generator=g, device=DEV).to(torch.bfloat16)
    _, _, dW13, dW2 = layer.backward(dy, weight_grads=True)
    torch.cuda.synchronize()
    assert L.check_status(layer.dev_status) == 0
    k, d, F = cfg.k, cfg.d, cfg.F
    counts = layer.counts.cpu().numpy()
    offsets = layer.offsets.cpu().numpy()
    nz = np.nonzero(counts)[0]
    experts = [int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])])]
    s2s = layer.s2s.cpu().numpy()
    sl2 = layer.sl2.cpu().numpy()
    for e in experts:
        rows = np.arange(offsets[e], offsets[e + 1])
        n = len(rows)
        tok = s2s[rows] // k
        slots = s2s[rows]
        xq, xs = oracle.quant_1x128(bf16_bits(x[torch.as_tensor(tok, device=DEV)]))
        re0 = np.zeros(n, np.int32)
        w13q, w13s = layer.w.w13_q[e:e + 1].cpu().numpy(), layer.w.w13_s[e:e + 1].cpu().numpy()
        w2q, w2s = layer.w.w2_q[e:e + 1].cpu().numpy(), layer.w.w2_s[e:e + 1].cpu().numpy()
        h = oracle.expert_ffn_preact(xq, xs, re0, w13q, w13s)
        act_f, _, _, out = oracle.expert_ffn(xq, xs, re0, w13q, w13s, w2q, w2s)
        gts = layer.gates.reshape(-1)[torch.as_tensor(slots, device=DEV)].cpu().numpy().reshape(n, 1)
        loc = np.arange(n, dtype=np.int32)
        d_out_f, dq, ds, _ = oracle.combine_backward(bf16_bits(dy[torch.as_tensor(tok, device=DEV)]), gts, out, loc)
        w2tq, w2ts = oracle.weight_transpose(w2q, w2s)
        d_act = oracle.grouped_gemm(dq, ds, re0, w2tq, w2ts)
        dh_f, _, _ = oracle.swiglu_backward(d_act, h)
        x_rows = bf16_to_f64(bf16_bits(x[torch.as_tensor(tok, device=DEV)])).astype(np.float32)
        off1 = np.array([0, n], np.int32)
        aq, as_, pad = oracle.quant_128x1(d_out_f, off1)
        bq, bs, _ = oracle.quant_128x1(act_f, off1)
        ref2 = oracle.wgrad(aq, as_, bq, bs, pad)[0]
        aq, as_, _ = oracle.quant_128x1(dh_f, off1)
        bq, bs, _ = oracle.quant_128x1(x_rows, off1)
        ref13 = oracle.wgrad(aq, as_, bq, bs, pad)[0]
        for got, ref, nm in ((dW2[e].cpu().numpy(), ref2, "dW2"), (dW13[e].cpu().numpy(), ref13, "dW13")):
            err = np.abs(got - ref).max() / np.abs(ref).max()
            assert err <= TOL, (nm, e, n, err)
        print(f"large wgrad: expert {e} ({n} rows) within {TOL}")
    empty = np.nonzero(counts == 0)[0]
    if len(empty):
        assert float(dW2[int(empty[0])].abs().max()) == 0.0


def test_wgrad_gemm_rejects_offsets_past_ld(L):
    """Padded offsets beyond the operands' ld are caught on the device: no
    tile runs (nothing is read past the scale arrays) and MOE_DEV_ROWS is
    set; the output of the experts with rows is left untouched."""
    E, M, N, ld = 2, 128, 128, 256
    a_q = torch.zeros((M, ld), dtype=torch.uint8, device=DEV)
    b_q = torch.zeros((N, ld), dtype=torch.uint8, device=DEV)
    a_sT = torch.ones((ld // 128, M), dtype=torch.float32, device=DEV)
    b_sT = torch.ones((ld // 128, N), dtype=torch.float32, device=DEV)
    pad = torch.tensor([0, 128, 384], dtype=torch.int32, device=DEV)
    out = torch.full((E, M, N), 7.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_wgrad_gemm(a_q, a_sT, b_q, b_sT, pad, out=out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & L.MOE_DEV_ROWS
    assert torch.all(out == 7.0)


def test_wgrad_quant_scales_off_the_fast_path(L, oracle):
    """The 128 x 1 x and g * dy legs where block scales leave the range the
    shared reciprocal serves (s < 2^-90: IEEE division), next to zero blocks
    (scale 1), bf16's largest values and ordinary ones, through a hand-built
    routing of 300 tokens over 3 experts: codes and scales bit-exact against
    the oracle."""
    T, k, E, d = 300, 2, 3, 256
    slots = np.arange(T * k)
    expert = (slots // k + slots % k) % E                     # two distinct experts per token
    s2s = np.argsort(expert, kind="stable").astype(np.int32)  # sorted row -> slot
    offsets = np.concatenate([[0], np.cumsum(np.bincount(expert, minlength=E))]).astype(np.int32)
    g = torch.Generator(device="cpu").manual_seed(11)
    xf = torch.randn((T, d), generator=g)
    xf[:, :64] *= 1e-30                                       # tiny blocks: s < 2^-90
    xf[:, 128:192] = 0.0                                      # zero blocks
    xf[::7, 192:] = 3.0e38                                    # bf16's largest values
    x = xf.to(torch.bfloat16)
    dy = torch.randn((T, d), generator=g).to(torch.bfloat16)
    gates = torch.rand((T, k), generator=g) + 0.1
    gates.view(-1)[torch.from_numpy(expert == 1)] = 1e-35     # expert 1's g * dy blocks tiny
    dev_offsets = torch.from_numpy(offsets).to(DEV)
    dev_s2s = torch.from_numpy(s2s).to(DEV)
    pad = L.moe_wgrad_pad_offsets(dev_offsets)
    ld = L.wgrad_ld(T * k, E)
    x_rows = bf16_to_f64(bf16_bits(x)).astype(np.float32)[s2s // k]
    dy_rows = bf16_to_f64(bf16_bits(dy)).astype(np.float32)[s2s // k]
    gdy_rows = gates.numpy().reshape(-1)[s2s][:, None].astype(np.float32) * dy_rows   # RN(g * dy)
    for src, kw, rows in ((L.WGRAD_SRC_X, dict(x=x.to(DEV)), x_rows),
                          (L.WGRAD_SRC_GDY, dict(dy=dy.to(DEV), gates=gates.to(DEV)), gdy_rows)):
        q, s = L.moe_wgrad_quant(src, dev_offsets, pad, d, ld, True, sorted_to_slot=dev_s2s, k=k, **kw)
        oq, os_, opad = oracle.quant_128x1(rows, offsets)
        P = int(opad[-1])
        assert (os_ < 2.0 ** -90).any()                       # the IEEE path is exercised
        np.testing.assert_array_equal(q.cpu().numpy()[:, :P], oq)
        np.testing.assert_array_equal(s.cpu().numpy()[:P // 128].T.view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("name,T", [("tiny", None), ("replay", 500)])
def test_layer_router_backward(L, oracle, name, T):
    """layer.router_backward on the d_gates of layer.backward: the router's
    dx and dW_r for the forward's ids (routed, or replayed from the payload)
    against the oracle's (1e-4 of the largest entry: the gate derivative is
    fp32 on the device)."""
    cfg = S.CONFIGS[name]
    if T:
        cfg = cfg.with_(T=T)
    layer = _layer(cfg)
    x = S.make_x(cfg, DEV)
    replay = S.make_replay_payload(cfg.with_(layers=1), DEV)[0] if cfg.mode == "replay" else None
    layer.forward(x, replay_kT=replay, train=True)
    g = torch.Generator(device=DEV).manual_seed(9)
    dy = torch.randn((cfg.T, cfg.d), generator=g, device=DEV).to(torch.bfloat16)
    _, d_gates = layer.backward(dy)
    dxr, dw = layer.router_backward(d_gates)
    torch.cuda.synchronize()
    assert L.check_status(layer.dev_status) == 0
    rdl, rdx, rdw = oracle.router_backward(bf16_bits(x), bf16_bits(layer.w.w_router), layer.ids[:cfg.T].cpu().numpy(),
                                           d_gates.cpu().numpy(), cfg.score_fn, cfg.renorm, cfg.route_scale)
    for got, ref in ((dxr, rdx), (dw, rdw)):
        assert np.abs(got.cpu().numpy() - ref).max() <= 1e-4 * np.abs(ref).max()
