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


# ------------------------------------------------------------------ weight gradients

def test_pad_offsets_hand_example(oracle):
    pad = oracle.pad_offsets(np.array([0, 1, 1, 129, 385, 512], np.int32))
    assert list(pad) == [0, 128, 128, 256, 512, 640]


def test_quant_128x1_against_torch(oracle):
    g = torch.Generator().manual_seed(13)
    offsets = np.array([0, 5, 5, 200, 330], np.int32)
    A, C = 330, 256
    x = (torch.randn(A, C, generator=g) * torch.exp2(torch.randint(-8, 8, (1, C), generator=g).float())).float()
    x[5:133, 7] = 0.0                                   # an all-zero block of one channel
    q, s, pad = oracle.quant_128x1(x.numpy(), offsets)
    assert q.shape == (C, int(pad[-1])) and s.shape == (C, int(pad[-1]) // 128)
    for e in range(4):
        r0, rows = offsets[e], offsets[e + 1] - offsets[e]
        for b in range((rows + 127) // 128):
            n = min(128, rows - 128 * b)
            v = x[r0 + 128 * b: r0 + 128 * b + n].t()       # [C, n]
            amax = v.abs().amax(1)
            sref = amax / torch.tensor(448.0)
            sref[sref == 0] = 1.0
            kb = pad[e] // 128 + b
            np.testing.assert_array_equal(s[:, kb], sref.numpy())
            qref = (v / sref[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            np.testing.assert_array_equal(q[:, pad[e] + 128 * b: pad[e] + 128 * b + n], qref)
            assert np.all(q[:, pad[e] + 128 * b + n: pad[e] + 128 * b + 128] == 0)   # padding rows
    assert s[7, pad[2] // 128] == 1.0                 # the zero block of channel 7 (expert 2, first block)


def test_wgrad_against_float64(oracle):
    g = torch.Generator().manual_seed(17)
    offsets = np.array([0, 70, 70, 300], np.int32)
    A, M, N = 300, 256, 384
    a = torch.randn(A, M, generator=g).float()
    b = torch.randn(A, N, generator=g).float()
    aq, as_, pad = oracle.quant_128x1(a.numpy(), offsets)
    bq, bs, _ = oracle.quant_128x1(b.numpy(), offsets)
    out = oracle.wgrad(aq, as_, bq, bs, pad)
    deq = lambda q, s: e4m3_to_f64(q) * np.repeat(s.astype(np.float64), 128, axis=1)
    Ad, Bd = deq(aq, as_), deq(bq, bs)
    for e in range(3):
        seg = slice(pad[e], pad[e + 1])
        ref = Ad[:, seg] @ Bd[:, seg].T
        mag = np.abs(Ad[:, seg]) @ np.abs(Bd[:, seg]).T
        assert np.all(np.abs(out[e] - ref) <= mag * 2.0 ** -20 + 1e-30)
    assert np.all(out[1] == 0)                          # the expert with no rows


def test_weight_gradients_dense_against_autograd(oracle):
    """E = 1: dW2 = d_out^T act and dW13 = dh^T x of a dense SwiGLU layer,
    from the 128 x 1 quantised operands, against float64 autograd."""
    cfg = S.CONFIGS["tiny"]
    n = 200
    g = torch.Generator().manual_seed(19)
    x = torch.randn(n, cfg.d, generator=g).double()
    W13 = (torch.randn(2 * cfg.F, cfg.d, generator=g) * 0.02).double().requires_grad_(True)
    W2 = (torch.randn(cfg.d, cfg.F, generator=g) * 0.02).double().requires_grad_(True)
    h = x @ W13.T
    act = torch.nn.functional.silu(h[:, :cfg.F]) * h[:, cfg.F:]
    act.retain_grad()
    h.retain_grad()
    y = act @ W2.T
    dy = torch.randn(n, cfg.d, generator=g).double()
    y.backward(dy)
    offsets = np.array([0, n], np.int32)
    dq, ds, pad = oracle.quant_128x1(dy.float().numpy(), offsets)
    aq, as_, _ = oracle.quant_128x1(act.detach().float().numpy(), offsets)
    dW2 = oracle.wgrad(dq, ds, aq, as_, pad)[0]
    hq, hs, _ = oracle.quant_128x1(h.grad.float().numpy(), offsets)
    xq, xs, _ = oracle.quant_128x1(x.float().numpy(), offsets)
    dW13 = oracle.wgrad(hq, hs, xq, xs, pad)[0]
    rel = lambda a, b: np.abs(a - b).max() / np.abs(b).max()
    # two e4m3 operands per product: a few percent of the largest entry
    assert rel(dW2, W2.grad.numpy()) < 5e-2, rel(dW2, W2.grad.numpy())
    assert rel(dW13, W13.grad.numpy()) < 5e-2, rel(dW13, W13.grad.numpy())
