"""GPU parity of the gathered form of the layer (GEMM1 A rows gathered from
the token-major codes by tile::gather4, GEMM2 outputs stored in slot order,
slot-order combine) against the CPU oracle, and bit-identity with the
sorted form (dispatch row copy, sorted outputs) on the same inputs."""
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


def _layers(cfg, T_max=None):
    from block_scaled_fp8_router_gb300.layer import MoELayerFP8, MoEWeightsFP8, quantize_weights
    wr = S.make_router_w(cfg, DEV)
    w13, w2 = S.make_w13(cfg, DEV), S.make_w2(cfg, DEV)
    w = MoEWeightsFP8(wr, *quantize_weights(w13, w2))
    T_max = T_max or cfg.T
    a = MoELayerFP8(w, T_max, cfg.k, cfg.score_fn, gathered=False)
    b = MoELayerFP8(w, T_max, cfg.k, cfg.score_fn, gathered=True)
    return a, b, w13, w2


def _check_same(L, a, b, T, k):
    A = T * k
    sl2 = a.sl2[:A]
    routed = sl2 >= 0
    # slot-order outputs are the sorted outputs, permuted
    assert torch.equal(b.out_sorted[:A][routed].view(torch.int16),
                       a.out_sorted[:A][sl2[routed].long()].view(torch.int16))
    assert torch.equal(a.y[:T].view(torch.int16), b.y[:T].view(torch.int16))
    assert L.check_status(a.dev_status) == 0 and L.check_status(b.dev_status) == 0


@pytest.mark.parametrize("name,T", [("tiny", None), ("replay", 700), ("large", 300)])
def test_gathered_equals_sorted(L, name, T):
    cfg = S.CONFIGS[name]
    if T:
        cfg = cfg.with_(T=T)
    a, b, _, _ = _layers(cfg)
    x = S.make_x(cfg, DEV)
    replay = S.make_replay_payload(cfg.with_(layers=1), DEV)[0] if cfg.mode == "replay" else None
    a.forward(x, replay_kT=replay)
    b.forward(x, replay_kT=replay)
    torch.cuda.synchronize()
    _check_same(L, a, b, cfg.T, cfg.k)


@pytest.mark.parametrize("name", ["tiny", "replay"])
def test_gathered_layer_against_oracle(L, oracle, name):
    """Every token of the gathered layer against the oracle's composition
    route/replay -> quant -> dispatch -> expert FFN -> combine."""
    cfg = S.CONFIGS[name]
    _, b, w13, w2 = _layers(cfg)
    x = S.make_x(cfg, DEV)
    replay = S.make_replay_payload(cfg, DEV)[0] if cfg.mode == "replay" else None
    y = b.forward(x, replay_kT=replay)
    torch.cuda.synchronize()
    assert L.check_status(b.dev_status) == 0
    xb = bf16_bits(x)
    l = oracle.router_logits(xb, bf16_bits(b.w.w_router))
    ids = oracle.topk(l, cfg.k) if replay is None else oracle.replay(replay.cpu().numpy(), cfg.E)[0]
    g = oracle.gates(l, ids, cfg.score_fn, cfg.renorm, cfg.route_scale)
    counts, offsets, s2s, sl2, _ = oracle.dispatch(ids, cfg.E)
    np.testing.assert_array_equal(b.s2s.cpu().numpy(), s2s)
    xq, xs = oracle.quant_1x128(xb)
    A = cfg.T * cfg.k
    row_e = np.repeat(np.arange(cfg.E, dtype=np.int32), counts)
    w13q, w13s = oracle.quant_128x128(bf16_bits(w13.reshape(-1, cfg.d)))
    w2q, w2s = oracle.quant_128x128(bf16_bits(w2.reshape(-1, cfg.F)))
    w = (w13q.reshape(cfg.E, 2 * cfg.F, cfg.d), w13s.reshape(cfg.E, 2 * cfg.F // 128, cfg.d // 128),
         w2q.reshape(cfg.E, cfg.d, cfg.F), w2s.reshape(cfg.E, cfg.d // 128, cfg.F // 128))
    _, _, _, out = oracle.expert_ffn(oracle.gather_rows(xq, s2s, A, cfg.k), oracle.gather_rows(xs, s2s, A, cfg.k),
                                     row_e, *w)
    # the gathered form keeps expert outputs in slot order
    out_slots = b.out_sorted[:A].cpu()
    routed = sl2 >= 0
    err_rows = row_rel_err(bf16_to_f64(bf16_bits(out_slots[torch.from_numpy(routed)])),
                           bf16_to_f64(out[sl2[routed]]))
    assert err_rows.max() <= TOL, err_rows.max()
    y_ref = oracle.combine(out, sl2, g)
    err = row_rel_err(bf16_to_f64(bf16_bits(y)), bf16_to_f64(y_ref))
    assert err.max() <= TOL, err.max()


def test_gathered_unrouted_slots_and_empty_experts(L):
    """Replayed ids with out-of-range entries (unrouted slots, skipped by the
    slot combine) and experts that receive no rows."""
    cfg = S.CONFIGS["replay"].with_(T=513)
    a, b, _, _ = _layers(cfg)
    x = S.make_x(cfg, DEV)
    p = S.make_replay_payload(cfg.with_(layers=1), DEV)[0].clone()
    p[p == 3] = 5            # expert 3 gets no rows (5 may now repeat within a token: flagged, gates 0)
    p[0, ::17] = cfg.E       # out of range: these slots are not routed
    a.forward(x, replay_kT=p)
    b.forward(x, replay_kT=p)
    torch.cuda.synchronize()
    assert int(a.counts[3]) == 0
    A = cfg.T * cfg.k
    assert torch.equal(a.y.view(torch.int16), b.y.view(torch.int16))
    sl2 = a.sl2[:A]
    routed = sl2 >= 0
    assert not bool(routed.all())
    assert torch.equal(b.out_sorted[:A][routed].view(torch.int16),
                       a.out_sorted[:A][sl2[routed].long()].view(torch.int16))


def test_gathered_full_size_equals_sorted(L):
    """The 8192-token large layer: gathered form == sorted form, bit for bit
    (the sorted form is checked against the oracle at this size elsewhere)."""
    cfg = S.CONFIGS["large"]
    a, b, _, _ = _layers(cfg)
    x = S.make_x(cfg, DEV)
    a.forward(x)
    b.forward(x)
    torch.cuda.synchronize()
    _check_same(L, a, b, cfg.T, cfg.k)


def test_gathered_out_of_range_slot_is_skipped(L):
    """A sorted_to_slot entry outside [0, T*k) marks its row as not routed:
    MOE_DEV_ROWS (0x4) is set, nothing is stored for it (guard rows on both
    sides of out_slots stay untouched) and every other slot's output equals
    the sorted form's."""
    cfg = S.CONFIGS["tiny"]
    a, _, _, _ = _layers(cfg)
    x = S.make_x(cfg, DEV)
    a.forward(x)
    torch.cuda.synchronize()
    T, k, d = cfg.T, cfg.k, cfg.d
    A = T * k
    s2s = a.s2s[:A].clone()
    bad_rows = [3, 10]
    lost = [int(s2s[r]) for r in bad_rows]
    s2s[3] = A + 7
    s2s[10] = -5
    guard = 32
    buf = torch.full((A + 2 * guard, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    out = buf[guard:guard + A]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    w = a.w
    L.moe_grouped_ffn_fp8_gathered(a.xq[:T], a.xs[:T], k, s2s, a.offsets, w.w13_q, w.w13_s, w.w2_q, w.w2_s,
                                   out_slots=out, dev_status=st)
    torch.cuda.synchronize()
    assert L.check_status(st) & 0x4
    assert torch.isnan(buf[:guard].float()).all() and torch.isnan(buf[guard + A:].float()).all()
    sl2 = a.sl2[:A]
    keep = sl2 >= 0
    keep[lost] = False
    assert torch.isnan(out[lost].float()).all()
    assert torch.equal(out[keep].view(torch.int16), a.out_sorted[:A][sl2[keep].long()].view(torch.int16))
