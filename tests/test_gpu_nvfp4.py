"""GPU parity of the NVFP4 quantiser (fp8_quant_nvfp4) against the CPU
oracle, bit for bit: the packed E2M1 codes, the E4M3 block scales and the
tensor scale, on inputs with block magnitudes across the E4M3 scale range
(normal and subnormal block scales), all-zero blocks, signed zeros,
elements on E2M1 rounding midpoints, an all-zero tensor and an empty one."""
import numpy as np
import pytest
import torch

from tests.helpers import bf16_bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from block_scaled_fp8_router_gb300 import moe_r3
    return moe_r3


@pytest.fixture(scope="module")
def oracle():
    from oracle import oracle as O
    return O


def _input(rows, cols, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp2(
        torch.randint(-12, 7, (rows, cols // 16), generator=g).float()).repeat_interleave(16, dim=1)
    x[0, :16] = 0.0                                   # an all-zero block
    x[0, 16:32] = -0.0                                # signed zeros
    # a block whose scaled values sit on E2M1 midpoints: max 6 * 2^-3 = 0.75
    x[1, :16] = torch.tensor([0.75, 0.03125, 0.09375, 0.15625, 0.21875, 0.3125, 0.4375, 0.625,
                              -0.75, -0.03125, -0.09375, -0.15625, -0.21875, -0.3125, -0.4375, -0.625])
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("rows,cols,seed", [(1, 16, 1), (37, 272, 2), (256, 2048, 3), (1000, 7168, 4)])
def test_nvfp4_quant_bit_exact(L, oracle, rows, cols, seed):
    xb = _input(rows, cols, seed) if rows > 1 else torch.randn(rows, cols).to(torch.bfloat16)
    q, s, ts = L.fp8_quant_nvfp4(xb.to(DEV))
    torch.cuda.synchronize()
    oq, os_, oenc = oracle.quant_nvfp4(bf16_bits(xb))
    assert ts[0].item() == oenc
    assert ts[1].item() == xb.float().abs().max().item()
    np.testing.assert_array_equal(s.cpu().numpy(), os_)
    np.testing.assert_array_equal(q.cpu().numpy(), oq)


def test_nvfp4_quant_zero_and_empty(L, oracle):
    z = torch.zeros(4, 64, dtype=torch.bfloat16, device=DEV)
    q, s, ts = L.fp8_quant_nvfp4(z)
    torch.cuda.synchronize()
    assert ts[0].item() == 1.0 and ts[1].item() == 0.0
    assert torch.all(q == 0) and torch.all(s == 0)
    e = torch.zeros(0, 64, dtype=torch.bfloat16, device=DEV)
    q, s, ts = L.fp8_quant_nvfp4(e)
    torch.cuda.synchronize()
    assert q.shape == (0, 32) and s.shape == (0, 4) and ts[0].item() == 1.0


def test_nvfp4_quant_rounding_midpoints(L, oracle):
    """A tensor whose scales are exact (amax 0.75: s_enc = 3584, block scale
    448, element scale 8), so the scaled values 0.25, 0.75, ..., 5 sit on
    E2M1 rounding midpoints and the ties-to-even rule decides every code."""
    x = torch.zeros(2, 32)
    mid = torch.tensor([0.75, 0.03125, 0.09375, 0.15625, 0.21875, 0.3125, 0.4375, 0.625])
    x[1, :16] = torch.cat([mid, -mid])
    x[1, 16:32] = torch.cat([-mid, mid])
    xb = x.to(torch.bfloat16)
    q, s, ts = L.fp8_quant_nvfp4(xb.to(DEV))
    torch.cuda.synchronize()
    oq, os_, oenc = oracle.quant_nvfp4(bf16_bits(xb))
    assert oenc == 3584.0 and ts[0].item() == oenc
    np.testing.assert_array_equal(s.cpu().numpy(), os_)
    np.testing.assert_array_equal(q.cpu().numpy(), oq)


# ---------------------------------------------------------------------------
# The NVFP4 expert FFN (moe_grouped_ffn_nvfp4) against the oracle's NVFP4 mode
# (or_expert_ffn_nvfp4), every operand quantised by the oracle itself.  The
# tensor core accumulates the scaled FP4 products in fp32 (order unspecified)
# where the oracle sums them exactly, and act is rounded to bf16 and
# re-quantised, so a code can flip at a rounding midpoint; the bar is the
# layer's: per row max |gpu - oracle| / max |oracle| <= 2e-2.

from block_scaled_fp8_router_gb300 import synthetic as S   # noqa: E402
from tests.helpers import bf16_to_f64                      # noqa: E402

TOL = 2e-2


def _oracle_nvfp4_weights(oracle, w13, w2, experts):
    q13, s13, e13, q2, s2, e2 = [], [], [], [], [], []
    for e in experts:
        q, s, enc = oracle.quant_nvfp4(bf16_bits(w13[e])); q13.append(q); s13.append(s); e13.append(enc)
        q, s, enc = oracle.quant_nvfp4(bf16_bits(w2[e])); q2.append(q); s2.append(s); e2.append(enc)
    return (np.stack(q13), np.stack(s13), np.array(e13, np.float32), np.stack(q2), np.stack(s2),
            np.array(e2, np.float32))


@pytest.mark.parametrize("counts,d,F", [
    ([128], 128, 128),                        # half K blocks in both GEMMs, d % 256 == 128 N tail
    ([1, 127, 128, 129, 300, 0, 5], 256, 256),
    ([0, 0, 200, 0], 256, 384),               # GEMM2 K = 384: a half last K block
    ([260, 3, 0, 64], 384, 256),              # GEMM1 half K block, GEMM2 N tail
])
def test_grouped_ffn_nvfp4_against_oracle(L, oracle, parity_report, counts, d, F):
    from block_scaled_fp8_router_gb300.layer import quantize_weights_nvfp4
    E = len(counts)
    A = int(sum(counts))
    cfg = S.CONFIGS["tiny"].with_(d=d, F=F, E=E, w_std=0.02)
    w13 = torch.stack([S.make_w13_expert(cfg, e, DEV, 5) for e in range(E)])
    w2 = torch.stack([S.make_w2_expert(cfg, e, DEV, 5) for e in range(E)])
    W = quantize_weights_nvfp4(None, w13, w2)
    g = torch.Generator(device=DEV).manual_seed(len(counts) + d)
    x = torch.randn((A, d), generator=g, device=DEV).to(torch.bfloat16)
    xq, xs, xts = L.fp8_quant_nvfp4(x)
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device=DEV)
    ws = torch.zeros(L.moe_grouped_ffn_nvfp4_workspace_size(A, d, F), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = L.moe_grouped_ffn_nvfp4(xq, xs, xts, offsets, W.w13_q, W.w13_sf, W.w13_enc, W.w2_q, W.w2_sf, W.w2_enc,
                                  workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert L.check_status(st) == 0
    ow = _oracle_nvfp4_weights(oracle, w13, w2, range(E))
    np.testing.assert_array_equal(W.w13_q.cpu().numpy(), ow[0])      # the weights' codes, scales and
    np.testing.assert_array_equal(W.w2_s.cpu().numpy(), ow[4])       # tensor scales are bit-exact
    np.testing.assert_array_equal(W.w13_enc.cpu().numpy(), ow[2])
    oq, os_, oenc = oracle.quant_nvfp4(bf16_bits(x))
    row_e = np.repeat(np.arange(E, dtype=np.int32), counts)
    _, act, _, _, _, ref = oracle.expert_ffn_nvfp4(oq, os_, oenc, row_e, *ow)
    g_act = ws[: A * F * 2].view(torch.bfloat16).view(A, F)
    assert parity_report(f"nvfp4 act {counts[:3]}.. d={d} F={F}", bf16_to_f64(bf16_bits(g_act)),
                         bf16_to_f64(act)).max() <= TOL
    err = parity_report(f"nvfp4 out {counts[:3]}.. d={d} F={F}", bf16_to_f64(bf16_bits(out)), bf16_to_f64(ref))
    assert err.max() <= TOL, err.max()


def test_nvfp4_tiled_scales_layout(L):
    """The scale images: word (g, kb, m, r, q) = scale bytes 16kb + 4m .. +3 of
    row 128g + 32q + r, zero past the row (checked against a numpy
    rearrangement of random bytes, K with a half last block)."""
    rows, K = 256, 384
    s = torch.randint(0, 256, (rows, K // 16), dtype=torch.uint8, device=DEV)
    t = L.moe_nvfp4_tile_scales(s, K).cpu().numpy()
    sn = s.cpu().numpy()
    nkb = (K + 255) // 256
    pad = np.zeros((rows, nkb * 16), np.uint8)
    pad[:, : K // 16] = sn
    ref = pad.reshape(rows // 128, 4, 32, nkb, 4, 4)            # [g, q, r, kb, m, byte]
    ref = ref.transpose(0, 3, 4, 2, 1, 5).reshape(-1)          # [g, kb, m, r, q, byte]
    np.testing.assert_array_equal(t, ref)


@pytest.mark.parametrize("name,T,E", [("tiny", None, None), ("replay", 64, None), ("large", 16, 16)])
def test_nvfp4_layer_against_oracle(L, oracle, parity_report, name, T, E):
    """The composed NVFP4 layer (route or replay -> NVFP4 x -> dispatch -> FFN
    -> combine) against the oracle, every token: tiny, the router-replay shape
    (64 tokens) and the large per-expert shape (d=7168, F=2048, top-8; 16
    tokens, 16 experts).  The token counts are small because the oracle sums
    every NVFP4 product exactly in float64 (a few rows per second at d=7168)."""
    from block_scaled_fp8_router_gb300.layer import MoELayerNVFP4, quantize_weights_nvfp4
    cfg = S.CONFIGS[name]
    if T:
        cfg = cfg.with_(T=T)
    if E:
        cfg = cfg.with_(E=E)
    x = S.make_x(cfg, DEV)
    wr = S.make_router_w(cfg, DEV)
    w13, w2 = S.make_w13(cfg, DEV), S.make_w2(cfg, DEV)
    W = quantize_weights_nvfp4(wr, w13, w2)
    layer = MoELayerNVFP4(W, cfg.T, cfg.k, cfg.score_fn, cfg.renorm, cfg.route_scale)
    replay = S.make_replay_payload(cfg.with_(layers=1), DEV)[0] if cfg.mode == "replay" else None
    y = layer.forward(x, replay_kT=replay)
    torch.cuda.synchronize()
    assert L.check_status(layer.dev_status) == 0
    xb = bf16_bits(x)
    lg = oracle.router_logits(xb, bf16_bits(wr))
    ids = oracle.topk(lg, cfg.k) if replay is None else oracle.replay(replay.cpu().numpy(), cfg.E)[0]
    np.testing.assert_array_equal(layer.ids.cpu().numpy(), ids)
    gts = oracle.gates(lg, ids, cfg.score_fn, cfg.renorm, cfg.route_scale)
    counts, offsets, s2s, sl2, _ = oracle.dispatch(ids, cfg.E)
    np.testing.assert_array_equal(layer.offsets.cpu().numpy(), offsets)
    A = cfg.T * cfg.k
    oq, os_, oenc = oracle.quant_nvfp4(xb)
    assert layer.x_ts[0].item() == oenc
    np.testing.assert_array_equal(layer.xq_sorted[:A].cpu().numpy(), oracle.gather_rows(oq, s2s, A, cfg.k))
    used = np.nonzero(counts)[0]
    remap = np.full(cfg.E, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    ow = _oracle_nvfp4_weights(oracle, w13, w2, used)
    row_e = remap[np.repeat(np.arange(cfg.E, dtype=np.int32), counts)]
    _, _, _, _, _, out = oracle.expert_ffn_nvfp4(oracle.gather_rows(oq, s2s, A, cfg.k),
                                                 oracle.gather_rows(os_, s2s, A, cfg.k), oenc, row_e, *ow)
    y_ref = oracle.combine(out, sl2, gts)
    err = parity_report(f"nvfp4 {name} layer y, all tokens", bf16_to_f64(bf16_bits(y)), bf16_to_f64(y_ref))
    assert err.max() <= TOL, err.max()
