"""GPU parity of the grouped block-scaled FP8 SwiGLU FFN (tcgen05) and of the
composed layer against the CPU oracle.

The GEMMs accumulate each 128-deep block in the tensor core (fp32, order not
specified) where the oracle sums it exactly, so act and out agree to fp32
rounding, and the 1x128 requantisation of act may flip a code where act/s
sits on a rounding midpoint.  Bar: per row, max |gpu - oracle| / max |oracle|
<= 2e-2 (the layer's contract); the measured error is far below it."""
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


def _weights(L, cfg, experts, seed=0):
    w13 = torch.stack([S.make_w13_expert(cfg, e, DEV, seed) for e in experts])
    w2 = torch.stack([S.make_w2_expert(cfg, e, DEV, seed) for e in experts])
    from block_scaled_fp8_router_gb300.layer import quantize_weights
    return w13, w2, quantize_weights(w13, w2)


def _oracle_weights(oracle, w13, w2):
    q13, s13, q2, s2 = [], [], [], []
    for e in range(w13.shape[0]):
        q, s = oracle.quant_128x128(bf16_bits(w13[e])); q13.append(q); s13.append(s)
        q, s = oracle.quant_128x128(bf16_bits(w2[e])); q2.append(q); s2.append(s)
    return np.stack(q13), np.stack(s13), np.stack(q2), np.stack(s2)


def _run_ffn(L, counts, d, F, seed=0, max_rows=None, x_std=1.0):
    E = len(counts)
    cfg = S.CONFIGS["tiny"].with_(d=d, F=F, E=E, w_std=0.02)
    w13, w2, (w13_q, w13_s, w2_q, w2_s) = _weights(L, cfg, range(E), seed)
    A = int(sum(counts))
    mr = max(A, 1) if max_rows is None else max_rows
    g = torch.Generator(device=DEV).manual_seed(seed + 1)
    x = (torch.randn((max(A, mr), d), generator=g, device=DEV) * x_std).to(torch.bfloat16)
    xq, xs = L.fp8_block_quant(x, 1)
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device=DEV)
    out = torch.full((mr, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(L.moe_grouped_ffn_workspace_size(mr, d, F), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_grouped_ffn_fp8(xq[:mr], xs[:mr], offsets, w13_q, w13_s, w2_q, w2_s, out_sorted=out, workspace=ws,
                          dev_status=st)
    torch.cuda.synchronize()
    return dict(x=x, xq=xq, xs=xs, w13=w13, w2=w2, out=out, ws=ws, st=L.check_status(st), A=A, mr=mr,
                counts=counts)


def _oracle_ffn(oracle, r, rows):
    counts = r["counts"]
    row_e = np.repeat(np.arange(len(counts), dtype=np.int32), counts)[rows]
    w = _oracle_weights(oracle, r["w13"], r["w2"])
    xq, xs = oracle.quant_1x128(bf16_bits(r["x"][rows]))
    return oracle.expert_ffn(xq, xs, row_e, *w)


@pytest.mark.parametrize("counts,d,F", [
    ([128], 128, 128),
    ([1, 127, 128, 129, 300, 0, 5], 256, 256),
    ([0, 0, 200, 0], 256, 384),
    ([260, 3, 0, 64], 384, 256),          # d % 256 == 128: GEMM2 N tail
])
def test_grouped_ffn_against_oracle(L, oracle, parity_report, counts, d, F):
    r = _run_ffn(L, counts, d, F, seed=len(counts) + d)
    assert r["st"] == 0
    A = r["A"]
    act_f, act_q, act_s, out = _oracle_ffn(oracle, r, np.arange(A))
    # act (dequantised from the workspace) against the oracle's act
    ws = r["ws"].cpu().numpy()
    g_actq = ws[: A * F].reshape(A, F)
    off = (r["mr"] * F + 255) // 256 * 256
    g_acts = ws[off: off + A * (F // 128) * 4].view(np.float32).reshape(A, F // 128)
    g_act = e4m3_to_f64(g_actq) * np.repeat(g_acts.astype(np.float64), 128, axis=1)
    ref_act = e4m3_to_f64(act_q) * np.repeat(act_s.astype(np.float64), 128, axis=1)
    assert parity_report(f"act {counts[:3]}.. d={d} F={F}", g_act, ref_act).max() <= TOL
    flips = (g_actq != act_q).mean()
    assert flips < 1e-2, flips
    err = parity_report(f"out {counts[:3]}.. d={d} F={F}", bf16_to_f64(bf16_bits(r["out"][:A])), bf16_to_f64(out))
    assert err.max() <= TOL, err.max()
    print(f"counts={counts} d={d} F={F}: max row rel err {err.max():.2e}, act code flips {flips:.1e}")


def test_grouped_ffn_row_bound(L, oracle):
    """expert_offsets[E] beyond max_rows: flagged, the clipped rows are still
    right, nothing past max_rows is written."""
    r = _run_ffn(L, [100, 100], 256, 256, max_rows=150)
    assert r["st"] & 0x4
    _, _, _, out = _oracle_ffn(oracle, r, np.arange(150))
    err = row_rel_err(bf16_to_f64(bf16_bits(r["out"][:150])), bf16_to_f64(out))
    assert err.max() <= TOL


def test_grouped_ffn_all_empty(L):
    r = _run_ffn(L, [0, 0, 0], 256, 256, max_rows=8)
    assert r["st"] == 0
    assert torch.isnan(r["out"].float()).all()      # nothing written


def test_grouped_ffn_no_rows(L):
    """max_rows = 0: the call launches nothing and accepts the empty
    tensors' NULL pointers, an empty workspace included."""
    r = _run_ffn(L, [0, 0, 0], 256, 256, max_rows=0)
    assert r["st"] == 0 and r["out"].shape == (0, 256) and r["ws"].numel() == 0


@pytest.mark.parametrize("name", ["tiny", "replay"])
def test_layer_against_oracle(L, oracle, parity_report, name):
    """The composed layer (route or replay -> quant -> dispatch -> FFN ->
    combine) on the tiny and router-replay workloads, every token checked."""
    from block_scaled_fp8_router_gb300.layer import MoELayerFP8, MoEWeightsFP8, quantize_weights
    cfg = S.CONFIGS[name]
    x = S.make_x(cfg, DEV)
    wr = S.make_router_w(cfg, DEV)
    w13, w2 = S.make_w13(cfg, DEV), S.make_w2(cfg, DEV)
    layer = MoELayerFP8(MoEWeightsFP8(wr, *quantize_weights(w13, w2)), cfg.T, cfg.k, cfg.score_fn)
    replay = S.make_replay_payload(cfg, DEV)[0] if cfg.mode == "replay" else None
    y = layer.forward(x, replay_kT=replay)
    torch.cuda.synchronize()
    assert L.check_status(layer.dev_status) == 0
    xb = bf16_bits(x)
    l = oracle.router_logits(xb, bf16_bits(wr))
    if replay is None:
        ids = oracle.topk(l, cfg.k)
    else:
        ids, _, _ = oracle.replay(replay.cpu().numpy(), cfg.E)
    np.testing.assert_array_equal(layer.ids.cpu().numpy(), ids)
    g = oracle.gates(l, ids, cfg.score_fn, cfg.renorm, cfg.route_scale)
    counts, offsets, s2s, sl2, _ = oracle.dispatch(ids, cfg.E)
    np.testing.assert_array_equal(layer.offsets.cpu().numpy(), offsets)
    np.testing.assert_array_equal(layer.sl2.cpu().numpy(), sl2)
    xq, xs = oracle.quant_1x128(xb)
    np.testing.assert_array_equal(layer.xq.cpu().numpy(), xq)
    A = cfg.T * cfg.k
    np.testing.assert_array_equal(layer.xq_sorted.cpu().numpy(), oracle.gather_rows(xq, s2s, A, cfg.k))
    row_e = np.repeat(np.arange(cfg.E, dtype=np.int32), counts)
    w = _oracle_weights(oracle, w13, w2)
    np.testing.assert_array_equal(layer.w.w13_q.cpu().numpy(), w[0])
    np.testing.assert_array_equal(layer.w.w2_s.cpu().numpy(), w[3])
    _, _, _, out = oracle.expert_ffn(oracle.gather_rows(xq, s2s, A, cfg.k), oracle.gather_rows(xs, s2s, A, cfg.k),
                                     row_e, *w)
    y_ref = oracle.combine(out, sl2, g)
    err = parity_report(f"{name} layer y, all tokens", bf16_to_f64(bf16_bits(y)), bf16_to_f64(y_ref))
    assert err.max() <= TOL, err.max()


def test_grouped_ffn_negative_offset_is_clipped(L, oracle):
    """An expert offset below 0 is clipped to row 0 and flagged
    (MOE_DEV_ROWS = 0x4): guard rows on both sides of the output and guard
    bytes before the workspace stay untouched, and the rows inside are the
    clipped experts' outputs."""
    d, F, E, mr, guard = 256, 256, 2, 200, 64
    cfg = S.CONFIGS["tiny"].with_(d=d, F=F, E=E, w_std=0.02)
    w13, w2, (w13_q, w13_s, w2_q, w2_s) = _weights(L, cfg, range(E), 3)
    g = torch.Generator(device=DEV).manual_seed(4)
    x = torch.randn((mr, d), generator=g, device=DEV).to(torch.bfloat16)
    xq, xs = L.fp8_block_quant(x, 1)
    offsets = torch.tensor([-50, 100, 200], dtype=torch.int32, device=DEV)
    buf = torch.full((mr + 2 * guard, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    out = buf[guard:guard + mr]
    need = L.moe_grouped_ffn_workspace_size(mr, d, F)
    ws_buf = torch.full((need + 2 * 4096,), 0xAB, dtype=torch.uint8, device=DEV)
    ws = ws_buf[4096:4096 + need]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_grouped_ffn_fp8(xq, xs, offsets, w13_q, w13_s, w2_q, w2_s, out_sorted=out, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert L.check_status(st) & 0x4
    assert torch.isnan(buf[:guard].float()).all() and torch.isnan(buf[guard + mr:].float()).all()
    assert (ws_buf[:4096] == 0xAB).all() and (ws_buf[4096 + need:] == 0xAB).all()
    _, _, _, ref = _oracle_ffn(oracle, dict(x=x, w13=w13, w2=w2, counts=[100, 100]), np.arange(mr))
    err = row_rel_err(bf16_to_f64(bf16_bits(out)), bf16_to_f64(ref))
    assert err.max() <= TOL, err.max()
