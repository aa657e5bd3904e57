"""GPU parity of the SIMT kernels against the CPU oracle, through the C ABI:
quantiser codes/scales, router ids/logits/capture, replay, dispatch maps and
rows, combine -- all bit-exact; gates within 1e-5 relative."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_router_gb300 import synthetic as S
from tests.helpers import bf16_bits, bf16_to_f64

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from block_scaled_fp8_router_gb300 import moe_r3
    return moe_r3


# ------------------------------------------------------------------ quantiser

def _edge_rows(rows, cols, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn(rows, cols, generator=g, device=DEV)
    scale = torch.exp2(torch.randint(-30, 30, (rows, 1), generator=g, device=DEV).float())
    x = (x * scale).to(torch.bfloat16)
    if rows >= 6 and cols >= 256:
        x[0, :128] = 0.0
        x[1, 128:256] = -0.0
        x[2, :128] = 1e-40                       # bf16 subnormals
        x[3, :] = torch.linspace(-448 * 2.0 ** -9, 448 * 2.0 ** -9, cols, device=DEV).to(torch.bfloat16)
        x[4, :128] = 3.0e38
        x[5, :128] = 2.0 ** -130
    return x


@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 256), (300, 2048), (1031, 7168)])
def test_quant_1x128_bit_exact(L, oracle, rows, cols):
    x = _edge_rows(rows, cols, rows)
    q, s = L.fp8_block_quant(x, 1)
    rq, rs = oracle.quant_1x128(bf16_bits(x))
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    np.testing.assert_array_equal(q.cpu().numpy(), rq)


def test_quant_1x128_strided_source(L, oracle):
    big = _edge_rows(64, 512, 3)
    x = big[:, 128:384]                          # leading dimension 512
    q, s = L.fp8_block_quant(x, 1)
    rq, rs = oracle.quant_1x128(bf16_bits(x))
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)


def test_quant_1x128_division_sweep(L, oracle):
    """Every 61st positive bf16 value as a block amax, each block filled with
    every bf16 magnitude <= amax (alternating signs), 127 per block: the codes
    come from the scale's reciprocal and one correction step on the device,
    from IEEE division in the oracle -- bit-exact."""
    pos = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    blocks = []
    for i in range(0, len(pos), 61):
        v = pos[: i + 1].copy()
        v[1::2] *= -1
        for j in range(0, len(v), 127):
            blk = np.zeros(128, np.float32)
            blk[0] = pos[i]
            blk[1:1 + len(v[j:j + 127])] = v[j:j + 127]
            blocks.append(blk)
    cols = 7168
    per_row = cols // 128
    nrows = (len(blocks) + per_row - 1) // per_row
    flat = np.zeros((nrows * per_row, 128), np.float32)
    flat[: len(blocks)] = np.stack(blocks)
    x = torch.from_numpy(flat.reshape(nrows, cols)).to(torch.bfloat16).to(DEV)
    q, s = L.fp8_block_quant(x, 1)
    rq, rs = oracle.quant_1x128(bf16_bits(x))
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    np.testing.assert_array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("rows,cols", [(128, 128), (384, 256), (1408 * 2, 2048)])
def test_quant_128x128_bit_exact(L, oracle, rows, cols):
    w = _edge_rows(rows, cols, rows + cols)
    q, s = L.fp8_block_quant(w, 128)
    rq, rs = oracle.quant_128x128(bf16_bits(w))
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    np.testing.assert_array_equal(q.cpu().numpy(), rq)


def test_quant_large_weight_sampled(L, oracle):
    cfg = S.CONFIGS["large"]
    for e in (0, 255):
        w = S.make_w13_expert(cfg, e, DEV)
        q, s = L.fp8_block_quant(w, 128)
        rows = slice(128 * 7, 128 * 9)             # two block rows checked fully
        rq, rs = oracle.quant_128x128(bf16_bits(w[rows]))
        np.testing.assert_array_equal(q[rows].cpu().numpy(), rq)
        np.testing.assert_array_equal(s[7:9].cpu().numpy(), rs)


# ------------------------------------------------------------------ router

def _route_case(cfg, T=None, seed=0):
    x = S.make_x(cfg, DEV, seed, T=T)
    wr = S.make_router_w(cfg, DEV, seed)
    return x, wr


@pytest.mark.parametrize("name,T", [("tiny", None), ("replay", 1000), ("large", 200)])
def test_route_topk_bit_exact(L, oracle, name, T):
    cfg = S.CONFIGS[name]
    x, wr = _route_case(cfg, T)
    T = x.shape[0]
    cap = torch.full((cfg.k, T), -7, dtype=torch.int32, device=DEV)
    lg = torch.empty((T, cfg.E), dtype=torch.float32, device=DEV)
    ids, gates = L.moe_route_topk(x, wr, cfg.k, cfg.score_fn, cfg.renorm, cfg.route_scale,
                                  capture_kT=cap, logits_out=lg)
    rl = oracle.router_logits(bf16_bits(x), bf16_bits(wr))
    np.testing.assert_array_equal(lg.cpu().numpy().view(np.uint32), rl.view(np.uint32))
    rid = oracle.topk(rl, cfg.k)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_array_equal(cap.cpu().numpy(), rid.T)
    rg = oracle.gates(rl, rid, cfg.score_fn, cfg.renorm, cfg.route_scale)
    np.testing.assert_allclose(gates.cpu().numpy(), rg, rtol=1e-5, atol=0)


@pytest.mark.parametrize("score_fn,renorm,scale", [(0, 0, 1.0), (1, 0, 2.5), (0, 1, 0.5), (1, 1, 1.0)])
def test_route_topk_score_modes_and_ragged(L, oracle, score_fn, renorm, scale):
    cfg = S.CONFIGS["replay"].with_(E=300, d=384)    # two expert passes, ragged last pass
    x, wr = _route_case(cfg, 77, seed=5)
    ids, gates = L.moe_route_topk(x, wr, 7, score_fn, renorm, scale)
    rl = oracle.router_logits(bf16_bits(x), bf16_bits(wr))
    rid = oracle.topk(rl, 7)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(gates.cpu().numpy(), oracle.gates(rl, rid, score_fn, renorm, scale), rtol=1e-5)


def test_route_topk_ties(L, oracle):
    """Duplicate router rows give exactly equal logits: lower index first."""
    cfg = S.CONFIGS["tiny"].with_(E=64)
    x, wr = _route_case(cfg, 100, seed=9)
    wr[10] = wr[3]
    wr[40] = wr[3]
    wr[33] = wr[7]
    x[5] = 0.0                                   # all logits +0: ids 0..k-1
    ids, _ = L.moe_route_topk(x, wr, 6, 0, 1, 1.0)
    rid = oracle.topk(oracle.router_logits(bf16_bits(x), bf16_bits(wr)), 6)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    assert list(rid[5]) == [0, 1, 2, 3, 4, 5]


def test_route_topk_k_equals_E_and_k32(L, oracle):
    for E, k in [(8, 8), (64, 32), (1024, 32)]:
        cfg = S.CONFIGS["tiny"].with_(E=E)
        x, wr = _route_case(cfg, 40, seed=E)
        ids, gates = L.moe_route_topk(x, wr, k, 1, 1, 1.0)
        rl = oracle.router_logits(bf16_bits(x), bf16_bits(wr))
        rid = oracle.topk(rl, k)
        np.testing.assert_array_equal(ids.cpu().numpy(), rid)
        np.testing.assert_allclose(gates.cpu().numpy(), oracle.gates(rl, rid, 1, 1, 1.0), rtol=1e-5)


@pytest.mark.parametrize("T,E,d", [(8192, 256, 128), (4801, 250, 128), (9728, 256, 128), (16384, 256, 128),
                                   (3000, 512, 128), (13, 256, 256)])
def test_route_topk_token_blocks(L, oracle, T, E, d):
    """Token counts of one and two waves of clusters on 152 SMs (8192, 9728,
    16384), ragged token blocks (4801, 13: warps whose 8 tokens are partly
    or wholly past the end), four-CTA clusters (E = 512) and a ragged last
    expert CTA (E = 250): logits, ids and capture bit-exact."""
    cfg = S.CONFIGS["large"].with_(E=E, d=d)
    x, wr = _route_case(cfg, T, seed=T)
    lg = torch.empty((T, E), dtype=torch.float32, device=DEV)
    cap = torch.full((8, T), -7, dtype=torch.int32, device=DEV)
    ids, gates = L.moe_route_topk(x, wr, 8, 1, 1, 2.5, capture_kT=cap, logits_out=lg)
    rl = oracle.router_logits(bf16_bits(x), bf16_bits(wr))
    np.testing.assert_array_equal(lg.cpu().numpy().view(np.uint32), rl.view(np.uint32))
    rid = oracle.topk(rl, 8)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_array_equal(cap.cpu().numpy(), rid.T)
    np.testing.assert_allclose(gates.cpu().numpy(), oracle.gates(rl, rid, 1, 1, 2.5), rtol=1e-5, atol=0)


def test_route_empty(L):
    cfg = S.CONFIGS["tiny"]
    x = torch.empty((0, cfg.d), dtype=torch.bfloat16, device=DEV)
    ids, gates = L.moe_route_topk(x, S.make_router_w(cfg, DEV), 2, 0)
    assert ids.shape == (0, 2)


# ------------------------------------------------------------------ replay

def _offset_copy(t, offset):
    """t's values in a tensor that starts `offset` elements into its buffer."""
    if offset == 0:
        return t
    buf = torch.empty(t.numel() + offset, dtype=t.dtype, device=t.device)
    buf[offset:] = t.flatten()
    return buf[offset:].view(t.shape)


@pytest.mark.parametrize("k,offset", [(8, 0), (8, 8), (16, 0), (32, 8)])
def test_replay_copies_and_round_trips(L, oracle, k, offset):
    """Capture then replay: ids and gates bit for bit.  offset 8 puts x and
    W_r 16 bytes past a 32-byte boundary (the replay's 16-byte load path);
    k = 16 and 32 take four and eight threads per token."""
    cfg = S.CONFIGS["large"].with_(k=k)
    x, wr = _route_case(cfg, 300)
    x, wr = _offset_copy(x, offset), _offset_copy(wr, offset)
    cap = torch.empty((cfg.k, 300), dtype=torch.int32, device=DEV)
    ids, gates = L.moe_route_topk(x, wr, cfg.k, cfg.score_fn, 1, 1.0, capture_kT=cap)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    rids, rgates = L.moe_route_replay(cap, cfg.E, x, wr, cfg.score_fn, 1, 1.0, dev_status=st)
    assert torch.equal(rids, ids)
    assert torch.equal(rgates.view(torch.int32), gates.view(torch.int32))   # bit for bit
    assert L.check_status(st) == 0


@pytest.mark.parametrize("name", ["replay", "multilayer_replay"])
def test_replay_payload_against_oracle(L, oracle, name):
    cfg = S.CONFIGS[name].with_(T=2000, layers=2)
    payload = S.make_replay_payload(cfg, DEV)
    x, wr = _route_case(cfg, 2000)
    for l in range(2):
        slab = payload[l]
        ids, gates = L.moe_route_replay(slab, cfg.E, x, wr, cfg.score_fn, 1, 1.0)
        rid, valid, bad = oracle.replay(slab.cpu().numpy(), cfg.E)
        assert bad == 0
        np.testing.assert_array_equal(ids.cpu().numpy(), rid)
        rl = oracle.router_logits(bf16_bits(x), bf16_bits(wr))
        np.testing.assert_allclose(gates.cpu().numpy(), oracle.gates(rl, rid, cfg.score_fn, 1, 1.0), rtol=1e-5)


def test_replay_bad_ids_flagged(L, oracle):
    cfg = S.CONFIGS["tiny"]
    x, wr = _route_case(cfg, 64)
    p = torch.stack([torch.arange(64, device=DEV) % 8, (torch.arange(64, device=DEV) + 1) % 8]).to(torch.int32)
    p[0, 3] = 8          # out of range
    p[1, 9] = p[0, 9]    # duplicate
    p[0, 20] = -1
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids, gates = L.moe_route_replay(p, cfg.E, x, wr, 0, 1, 1.0, dev_status=st)
    assert L.check_status(st) & L.MOE_DEV_BAD_IDS
    rid, valid, bad = oracle.replay(p.cpu().numpy(), cfg.E)
    assert bad == 3
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    g = gates.cpu().numpy()
    assert np.all(g[valid == 0] == 0) and np.all(g[valid == 1].sum(1) > 0.99)
    # ids only (no x): no gates, still flags
    st.zero_()
    ids2, g2 = L.moe_route_replay(p, cfg.E, dev_status=st)
    assert g2 is None and torch.equal(ids2, ids) and L.check_status(st) & L.MOE_DEV_BAD_IDS


# ------------------------------------------------------------------ dispatch

def _check_dispatch(L, oracle, ids, E, rows=None, scales=None):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    counts, offsets, s2s, sl2, rs, ss = L.moe_dispatch(ids, E, rows=rows, row_scales=scales, dev_status=st)
    rc, ro, rs2s, rsl2, dropped = oracle.dispatch(ids.cpu().numpy(), E)
    n = int(ro[-1])
    np.testing.assert_array_equal(counts.cpu().numpy(), rc)
    np.testing.assert_array_equal(offsets.cpu().numpy(), ro)
    np.testing.assert_array_equal(s2s[:n].cpu().numpy(), rs2s[:n])
    np.testing.assert_array_equal(sl2.cpu().numpy(), rsl2)
    k = ids.shape[1]
    if rows is not None:
        ref = oracle.gather_rows(rows.cpu().contiguous().view(torch.uint8).numpy().reshape(rows.shape[0], -1),
                                 rs2s, n, k)
        got = rs[:n].cpu().contiguous().view(torch.uint8).numpy().reshape(n, -1)
        np.testing.assert_array_equal(got, ref)
    if scales is not None:
        np.testing.assert_array_equal(ss[:n].cpu().numpy(), oracle.gather_rows(scales.cpu().numpy(), rs2s, n, k))
    return L.check_status(st), dropped


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (129, 2, 8), (4096, 6, 64), (1500, 8, 256), (777, 32, 1024)])
def test_dispatch_maps_and_rows(L, oracle, T, k, E):
    g = torch.Generator(device=DEV).manual_seed(T)
    ids = torch.argsort(torch.rand((T, E), generator=g, device=DEV), dim=1)[:, :k].to(torch.int32)
    d = 256
    xq = torch.randint(0, 256, (T, d), generator=g, device=DEV, dtype=torch.uint8)
    xs = torch.rand((T, d // 128), generator=g, device=DEV)
    st, dropped = _check_dispatch(L, oracle, ids, E, xq, xs)
    assert st == 0 and dropped == 0


def test_dispatch_bf16_rows_skewed_with_empty_experts(L, oracle):
    cfg = S.CONFIGS["multilayer_replay"].with_(T=3000, d=384, layers=1)
    ids = S.make_replay_payload(cfg, DEV)[0].t().contiguous()
    x = S.make_x(cfg, DEV)
    st, _ = _check_dispatch(L, oracle, ids, cfg.E, x, None)
    assert st == 0


@pytest.mark.parametrize("T", [16384, 16385])
def test_dispatch_run_length_boundary(L, oracle, T):
    """E = 256, top-8: 131072 slots are the most the 128-slot warp runs take
    (their per-run counts fill 1 MiB); one more token switches to 1024-slot
    runs.  Maps and rows bit-exact on both sides."""
    cfg = S.CONFIGS["long_dispatch"].with_(T=T, d=128, layers=1)
    ids = S.make_replay_payload(cfg, DEV)[0].t().contiguous()
    x = S.make_x(cfg, DEV)
    st, dropped = _check_dispatch(L, oracle, ids, cfg.E, x, None)
    assert st == 0 and dropped == 0


def test_dispatch_bad_ids_dropped(L, oracle):
    ids = torch.tensor([[2, 9], [-1, 1], [0, 2], [3, 3]], dtype=torch.int32, device=DEV)
    x = torch.randn(4, 128, device=DEV).to(torch.bfloat16)
    st, dropped = _check_dispatch(L, oracle, ids, 4, x, None)
    assert dropped == 2 and st & 1


def test_dispatch_empty(L):
    ids = torch.empty((0, 4), dtype=torch.int32, device=DEV)
    counts, offsets, *_ = L.moe_dispatch(ids, 16)
    assert counts.sum().item() == 0 and offsets.cpu().tolist() == [0] * 17


# ------------------------------------------------------------------ combine

@pytest.mark.parametrize("T,k,d", [(1, 1, 128), (300, 6, 2048), (129, 32, 128), (64, 8, 7168)])
def test_combine_bit_exact(L, oracle, T, k, d):
    g = torch.Generator(device=DEV).manual_seed(T * k)
    out = torch.randn((T * k + 5, d), generator=g, device=DEV).to(torch.bfloat16)
    sl2 = torch.randperm(T * k, generator=g, device=DEV).to(torch.int32)
    sl2[::7] = -1
    gates = torch.rand((T, k), generator=g, device=DEV)
    y = L.moe_combine(out, sl2, gates)
    ref = oracle.combine(bf16_bits(out), sl2.cpu().numpy(), gates.cpu().numpy())
    np.testing.assert_array_equal(bf16_bits(y), ref)


def test_identity_experts_round_trip(L, oracle):
    """combine(dispatch(x)) == x for identity experts and Dirichlet gates."""
    cfg = S.CONFIGS["long_dispatch"].with_(T=5000)
    ids = S.make_replay_payload(cfg, DEV)[0].t().contiguous()
    gates = S.make_dirichlet_gates(cfg, DEV)
    x = S.make_x(cfg, DEV)
    counts, offsets, s2s, sl2, rows, _ = L.moe_dispatch(ids, cfg.E, rows=x)
    y = L.moe_combine(rows, sl2, gates)
    assert torch.equal(y.view(torch.int16), x.view(torch.int16))


# ------------------------------------------------------------------ faults

def test_bounded_wait_times_out(L):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_debug_bounded_wait(2_000_000, st)     # 2 ms, nothing ever arrives
    torch.cuda.synchronize()
    assert L.check_status(st) == L.MOE_DEV_TIMEOUT
    # the context is still usable
    y = torch.ones(4, device=DEV) * 2
    assert y.sum().item() == 8.0


def test_host_errors_raise(L):
    x = torch.zeros((4, 100), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(L.MoEError):
        L.fp8_block_quant(x, 1)


# ------------------------------------------------------------------ router backward

def _dispatch_maps(L, ids, E):
    T, k = ids.shape
    s2s = torch.empty(T * k, dtype=torch.int32, device=DEV)
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    L.moe_dispatch(ids, E, expert_offsets=offs, sorted_to_slot=s2s)
    return s2s, offs


@pytest.mark.parametrize("name,T,score_fn,renorm,rs", [("tiny", None, 0, 1, 1.0), ("replay", 1000, 0, 1, 2.0),
                                                       ("large", 300, 1, 1, 1.0), ("large", 257, 1, 0, 2.5)])
def test_router_backward_against_oracle(L, oracle, name, T, score_fn, renorm, rs):
    """d_logits against the oracle (the logits are the same fp32 chain; the
    gate derivative differs by fp32 vs double rounding); dx and dW_r against
    a float64 sum of the kernel's own d_logits within the fp32 summation
    bound n 2^-24 sum|terms|, and against the oracle's within 1e-4."""
    cfg = S.CONFIGS[name]
    x, wr = _route_case(cfg, T, seed=3)
    T, E, k, d = x.shape[0], cfg.E, cfg.k, cfg.d
    ids, _ = L.moe_route_topk(x, wr, k, score_fn, renorm, rs)
    g = torch.Generator(device=DEV).manual_seed(T)
    dg = torch.randn((T, k), generator=g, device=DEV)
    s2s, offs = _dispatch_maps(L, ids, E)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dl, dx, dw = L.moe_router_backward(x, wr, ids, dg, score_fn, renorm, rs, dx=True, dw_router=True,
                                       sorted_to_slot=s2s, expert_offsets=offs, dev_status=st)
    assert L.check_status(st) == 0
    rdl, rdx, rdw = oracle.router_backward(bf16_bits(x), bf16_bits(wr), ids.cpu().numpy(), dg.cpu().numpy(),
                                           score_fn, renorm, rs)
    dl_h = dl.cpu().numpy()
    assert np.abs(dl_h - rdl).max() <= 1e-5 * np.abs(rdl).max()
    xf = bf16_to_f64(bf16_bits(x))
    wf = bf16_to_f64(bf16_bits(wr))
    idn = ids.cpu().numpy()
    # dx: k terms per element
    terms = dl_h.astype(np.float64)[:, :, None] * wf[idn]                 # [T, k, d]
    ex, ab = terms.sum(1), np.abs(terms).sum(1)
    assert np.all(np.abs(dx.cpu().numpy() - ex) <= k * 2.0 ** -24 * ab + 1e-30)
    # dW_r: the rows of each expert
    onehot = np.zeros((E, T), np.float64)
    np.add.at(onehot, (idn.reshape(-1), np.repeat(np.arange(T), k)), dl_h.reshape(-1).astype(np.float64))
    absoh = np.zeros((E, T), np.float64)
    np.add.at(absoh, (idn.reshape(-1), np.repeat(np.arange(T), k)), np.abs(dl_h.reshape(-1)).astype(np.float64))
    ew, aw = onehot @ xf, absoh @ np.abs(xf)
    n_e = np.bincount(idn.reshape(-1), minlength=E)[:, None]
    assert np.all(np.abs(dw.cpu().numpy() - ew) <= n_e * 2.0 ** -24 * aw + 1e-30)
    for got, ref in ((dx, rdx), (dw, rdw)):
        assert np.abs(got.cpu().numpy() - ref).max() <= 1e-4 * np.abs(ref).max()


def test_router_backward_bad_ids_and_unchosen_experts(L, oracle):
    """A token with a repeated or out-of-range id gets zero d_logits (and
    sets the flag); experts nobody chose get zero dW_r rows."""
    cfg = S.CONFIGS["replay"].with_(E=70, d=256)
    x, wr = _route_case(cfg, 200, seed=8)
    T, k, E = 200, cfg.k, 70
    ids = torch.stack([torch.randperm(60)[:k] for _ in range(T)]).to(torch.int32).to(DEV)   # 60..69 unused
    ids[5, 1] = ids[5, 0]
    dg = torch.randn((T, k), device=DEV)
    s2s, offs = _dispatch_maps(L, ids, E)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dl, dx, dw = L.moe_router_backward(x, wr, ids, dg, 0, 1, 1.0, dw_router=True, sorted_to_slot=s2s,
                                       expert_offsets=offs, dev_status=st)
    assert L.check_status(st) & L.MOE_DEV_BAD_IDS
    assert torch.all(dl[5] == 0) and torch.all(dx[5] == 0)
    assert torch.all(dw[60:] == 0)
    valid = np.ones(T, np.uint8)
    valid[5] = 0
    rdl, _, rdw = oracle.router_backward(bf16_bits(x), bf16_bits(wr), ids.cpu().numpy(), dg.cpu().numpy(), 0, 1, 1.0,
                                         valid=valid)
    assert np.abs(dl.cpu().numpy() - rdl).max() <= 1e-5 * np.abs(rdl).max()
    assert np.abs(dw.cpu().numpy() - rdw).max() <= 1e-4 * np.abs(rdw).max()


def test_router_backward_clamps_bad_offsets(L):
    """Expert offsets that are negative, decreasing or past T*k are clamped
    into [0, T*k] (the kernel reads no row outside the map) and set
    MOE_DEV_ROWS; experts whose two offsets are intact keep their exact
    dW_r rows."""
    cfg = S.CONFIGS["replay"].with_(E=70, d=256)
    x, wr = _route_case(cfg, 200, seed=9)
    T, k, E = 200, cfg.k, 70
    ids = torch.stack([torch.randperm(E)[:k] for _ in range(T)]).to(torch.int32).to(DEV)
    dg = torch.randn((T, k), device=DEV)
    s2s, offs = _dispatch_maps(L, ids, E)
    _, _, dw_ref = L.moe_router_backward(x, wr, ids, dg, 0, 1, 1.0, dx=False, dw_router=True, sorted_to_slot=s2s,
                                         expert_offsets=offs)
    bad = offs.clone()
    bad[3] = -7                     # expert 2 ends before it starts, expert 3 starts before row 0
    bad[E] = T * k + 1000            # the last expert runs past the map
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    _, _, dw = L.moe_router_backward(x, wr, ids, dg, 0, 1, 1.0, dx=False, dw_router=True, sorted_to_slot=s2s,
                                     expert_offsets=bad, dev_status=st)
    torch.cuda.synchronize()
    assert L.check_status(st) == L.MOE_DEV_ROWS
    keep = [e for e in range(E) if e not in (2, 3, E - 1)]
    assert torch.equal(dw[keep], dw_ref[keep])
    assert torch.all(dw[2] == 0)    # an empty range after clamping


def test_router_backward_edge_cases(L, oracle):
    """T = 0 (empty tensors, dW_r zeroed); k = 1 under renormalisation (the
    gate is route_scale whatever the logit, so no gradient); k = 24 (eight
    threads per token in the logit pass) against the oracle; x and W_r 16
    bytes past a 32-byte boundary (the 16-byte load path) bit-identical to
    the aligned run."""
    cfg = S.CONFIGS["replay"].with_(E=64, d=256)
    E, d = 64, 256
    _, wr = _route_case(cfg, 8, seed=1)
    # T = 0
    x0 = torch.empty((0, d), dtype=torch.bfloat16, device=DEV)
    dw0 = torch.full((E, d), 7.0, device=DEV)
    dl, dx, dw = L.moe_router_backward(x0, wr, torch.empty((0, 6), dtype=torch.int32, device=DEV),
                                       torch.empty((0, 6), device=DEV), 1, 1, 1.0, dx=True, dw_router=dw0,
                                       sorted_to_slot=torch.empty(0, dtype=torch.int32, device=DEV),
                                       expert_offsets=torch.zeros(E + 1, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert dl.shape == (0, 6) and dx.shape == (0, d) and torch.all(dw == 0)
    # k = 1
    T = 130
    x, _ = _route_case(cfg, T, seed=2)
    ids1 = torch.randint(0, E, (T, 1), device=DEV, dtype=torch.int32)
    dg1 = torch.randn((T, 1), device=DEV)
    dl, dx, _ = L.moe_router_backward(x, wr, ids1, dg1, 0, 1, 1.0)
    assert torch.all(dl == 0) and torch.all(dx == 0)
    dl, _, _ = L.moe_router_backward(x, wr, ids1, dg1, 1, 1, 1.0)
    assert dl.abs().max().item() <= 1e-6 * dg1.abs().max().item()
    # k = 24, both alignments
    k = 24
    ids = torch.stack([torch.randperm(E)[:k] for _ in range(T)]).to(torch.int32).to(DEV)
    dg = torch.randn((T, k), device=DEV)
    s2s, offs = _dispatch_maps(L, ids, E)
    outs = []
    for off in (0, 8):
        xo, wro = _offset_copy(x, off), _offset_copy(wr, off)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        outs.append(L.moe_router_backward(xo, wro, ids, dg, 1, 1, 1.5, dx=True, dw_router=True,
                                          sorted_to_slot=s2s, expert_offsets=offs, dev_status=st))
        assert L.check_status(st) == 0
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    rdl, rdx, rdw = oracle.router_backward(bf16_bits(x), bf16_bits(wr), ids.cpu().numpy(), dg.cpu().numpy(), 1, 1,
                                           1.5)
    for got, ref, tol in zip(outs[0], (rdl, rdx, rdw), (1e-5, 1e-4, 1e-4)):
        assert np.abs(got.cpu().numpy() - ref).max() <= tol * np.abs(ref).max()
