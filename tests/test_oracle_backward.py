"""Pins for the oracle's backward of the expert path (the trainer replays
routing to train): combine, weight transpose, GEMM1 pre-activations, the
grouped GEMM used for dgrad, SwiGLU backward, dispatch backward.

- combine backward and SwiGLU backward against torch.autograd in float64
  (fp32 rounding of the oracle's results is the only difference), with
  quantised outputs checked against torch's e4m3 cast block by block;
- weight transpose: block quantisation commutes with transposition, so the
  transposed codes/scales equal the quantisation of the transposed bf16
  weights;
- GEMM1 pre-activations reproduce the forward's act through silu * up, and
  the grouped GEMM with (K, N) = (F, d) reproduces the forward's output bits;
- dispatch backward on integer-valued rows equals the exact sum;
- the whole expert-path backward on a dense E = 1 layer against autograd of
  the dequantised float64 forward.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_router_gb300 import synthetic as S
from tests.helpers import bf16_bits, bf16_to_f64, e4m3_to_f64, row_rel_err


def _bf16(a):
    return bf16_bits(torch.as_tensor(a, dtype=torch.float64).to(torch.bfloat16))


def _check_quant(v, q, s):
    """v [n, K] fp32 values, q codes, s [n, K/128] scales: the recipe's rule."""
    vb = torch.from_numpy(v.reshape(-1, 128))
    amax = vb.abs().amax(1)
    s_ref = amax / torch.tensor(448.0, dtype=torch.float32)
    s_ref[s_ref == 0] = 1.0
    np.testing.assert_array_equal(s.reshape(-1), s_ref.numpy())
    q_ref = (vb / s_ref[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(q.reshape(-1, 128), q_ref)


def test_combine_backward_against_autograd(oracle):
    g = torch.Generator().manual_seed(1)
    T, k, d = 37, 3, 256
    A = T * k
    perm = torch.randperm(A, generator=g)
    sl2 = perm.numpy().astype(np.int32)
    sl2[5] = -1                                      # one unrouted slot
    out = (torch.randn(A, d, generator=g)).to(torch.bfloat16)
    dy = (torch.randn(T, d, generator=g)).to(torch.bfloat16)
    gates = torch.rand(T, k, generator=g, dtype=torch.float32)
    d_out_f, d_out_q, d_out_s, d_g = oracle.combine_backward(bf16_bits(dy), gates.numpy(), bf16_bits(out), sl2)
    # autograd of y = sum_j g * out[r(t, j)] with upstream dy
    o64 = out.double().requires_grad_(True)
    g64 = gates.double().requires_grad_(True)
    idx = torch.from_numpy(np.where(sl2 >= 0, sl2, 0)).long()
    mask = torch.from_numpy(sl2 >= 0).double()
    y = (g64.reshape(-1, 1) * mask[:, None] * o64[idx]).reshape(T, k, d).sum(1)
    y.backward(dy.double())
    ref_dout = o64.grad.numpy()
    routed = sl2 >= 0
    assert np.all(np.abs(d_out_f[sl2[routed]] - ref_dout[sl2[routed]]) <= np.abs(ref_dout[sl2[routed]]) * 2.0 ** -24)
    ref_g = g64.grad.numpy()
    mag = (dy.double().abs()[:, None, :] * out.double().abs()[idx].reshape(T, k, d)).sum(2).numpy()
    assert np.all(np.abs(d_g - ref_g) <= mag * 2.0 ** -23)
    assert d_g.reshape(-1)[5] == 0.0
    _check_quant(d_out_f[sl2[routed]], d_out_q[sl2[routed]], d_out_s[sl2[routed]])


def test_weight_transpose_commutes_with_quantisation(oracle):
    cfg = S.CONFIGS["tiny"]
    w2 = torch.stack([S.make_w2_expert(cfg, e, "cpu") for e in range(3)])          # [E, d, F]
    q, s = [], []
    for e in range(3):
        a, b = oracle.quant_128x128(bf16_bits(w2[e]))
        q.append(a); s.append(b)
    qt, st = oracle.weight_transpose(np.stack(q), np.stack(s))
    for e in range(3):
        a, b = oracle.quant_128x128(bf16_bits(w2[e].t().contiguous()))
        np.testing.assert_array_equal(qt[e], a)
        np.testing.assert_array_equal(st[e], b)


def _expert_setup(oracle, cfg, n, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, cfg.d, generator=g).to(torch.bfloat16)
    xq, xs = oracle.quant_1x128(bf16_bits(x))
    w13q, w13s = oracle.quant_128x128(bf16_bits(S.make_w13_expert(cfg, 0, "cpu", seed)))
    w2q, w2s = oracle.quant_128x128(bf16_bits(S.make_w2_expert(cfg, 0, "cpu", seed)))
    return xq, xs, w13q[None], w13s[None], w2q[None], w2s[None]


def test_preact_and_grouped_gemm_reproduce_the_forward(oracle):
    cfg = S.CONFIGS["tiny"]
    xq, xs, w13q, w13s, w2q, w2s = _expert_setup(oracle, cfg, 24, 3)
    row_e = np.zeros(24, np.int32)
    act_f, act_q, act_s, out = oracle.expert_ffn(xq, xs, row_e, w13q, w13s, w2q, w2s)
    h = oracle.expert_ffn_preact(xq, xs, row_e, w13q, w13s).astype(np.float64)
    gte, up = h[:, :cfg.F], h[:, cfg.F:]
    act = (gte / (1 + np.exp(-gte))) * up
    assert np.all(np.abs(act.astype(np.float32) - act_f) <= np.abs(act) * 2.0 ** -23 + 1e-30)
    out2 = oracle.grouped_gemm(act_q, act_s, row_e, w2q, w2s)
    np.testing.assert_array_equal(out2, out)


def test_swiglu_backward_against_autograd(oracle):
    g = torch.Generator().manual_seed(7)
    n, F = 9, 256
    h = (torch.randn(n, 2 * F, generator=g) * 3).float()
    da = torch.randn(n, F, generator=g).to(torch.bfloat16)
    dh_f, dh_q, dh_s = oracle.swiglu_backward(bf16_bits(da), h.numpy())
    h64 = h.double().requires_grad_(True)
    act = torch.nn.functional.silu(h64[:, :F]) * h64[:, F:]
    act.backward(da.double())
    ref = h64.grad.numpy()
    assert np.all(np.abs(dh_f - ref) <= np.abs(ref) * 2.0 ** -23 + 1e-300)
    _check_quant(dh_f, dh_q, dh_s)


def test_dispatch_backward_exact_on_integers(oracle):
    g = torch.Generator().manual_seed(11)
    T, k, d = 21, 4, 128
    A = T * k
    sl2 = torch.randperm(A, generator=g).numpy().astype(np.int32)
    sl2[[3, 40]] = -1
    rows = torch.randint(-64, 64, (A, d), generator=g).to(torch.bfloat16)
    dx = oracle.dispatch_backward(bf16_bits(rows), sl2, T, k)
    r = rows.double().numpy()
    ref = np.zeros((T, d))
    for t in range(T):
        for j in range(k):
            if sl2[t * k + j] >= 0:
                ref[t] += r[sl2[t * k + j]]
    np.testing.assert_array_equal(bf16_to_f64(dx), ref)


def test_expert_backward_dense_against_autograd(oracle):
    """E = 1, k = 1, gate 1: the expert path's dX against autograd of the
    dequantised float64 forward (the e4m3 re-quantisation of the upstream
    gradient and of dh is the dominant difference)."""
    cfg = S.CONFIGS["tiny"]
    n = 16
    xq, xs, w13q, w13s, w2q, w2s = _expert_setup(oracle, cfg, n, 5)
    row_e = np.zeros(n, np.int32)
    act_f, act_q, act_s, out = oracle.expert_ffn(xq, xs, row_e, w13q, w13s, w2q, w2s)
    h = oracle.expert_ffn_preact(xq, xs, row_e, w13q, w13s)
    gq = torch.Generator().manual_seed(6)
    dy = torch.randn(n, cfg.d, generator=gq).to(torch.bfloat16)
    sl2 = np.arange(n, dtype=np.int32)
    _, d_out_q, d_out_s, _ = oracle.combine_backward(bf16_bits(dy), np.ones((n, 1), np.float32), out, sl2)
    w2tq, w2ts = oracle.weight_transpose(w2q, w2s)
    w13tq, w13ts = oracle.weight_transpose(w13q, w13s)
    d_act = oracle.grouped_gemm(d_out_q, d_out_s, row_e, w2tq, w2ts)
    _, dh_q, dh_s = oracle.swiglu_backward(d_act, h)
    dxs = oracle.grouped_gemm(dh_q, dh_s, row_e, w13tq, w13ts)
    dx = oracle.dispatch_backward(dxs, sl2, n, 1)
    # autograd of the dequantised forward (act not re-quantised)
    X = torch.from_numpy(e4m3_to_f64(xq) * np.repeat(xs.astype(np.float64), 128, axis=1)).requires_grad_(True)
    deq = lambda q, s: torch.from_numpy(e4m3_to_f64(q) * np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1))
    W13, W2 = deq(w13q[0], w13s[0]), deq(w2q[0], w2s[0])
    hh = X @ W13.T
    y = (torch.nn.functional.silu(hh[:, :cfg.F]) * hh[:, cfg.F:]) @ W2.T
    y.backward(dy.double())
    err = row_rel_err(bf16_to_f64(dx), X.grad.numpy())
    # two e4m3 re-quantisations (upstream gradient, dh): a few percent of the
    # row maximum; a dropped or misplaced term gives O(1)
    assert err.max() < 8e-2, err.max()
    # and the GEMMs themselves: d_act against float64 on the quantised operands
    Dq = torch.from_numpy(e4m3_to_f64(d_out_q) * np.repeat(d_out_s.astype(np.float64), 128, axis=1))
    ref_da = (Dq @ W2).numpy()
    got = bf16_to_f64(d_act)
    assert np.all(np.abs(got - ref_da) <= np.abs(ref_da) * 2.0 ** -8 + 1e-6 * np.abs(ref_da).max())
