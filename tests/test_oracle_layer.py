"""Pins for the oracle's dispatch, block-scaled GEMM, SwiGLU FFN and combine.

- dispatch: torch.bincount / cumsum / stable torch.sort; inverse bijection;
  brute force on tiny inputs; dropped out-of-range slots.
- GEMM: float64 torch.matmul on dequantised operands within the rounding
  bound of the per-block binary32 promotion chain.
- FFN: composition check (silu(gate) * up, 1x128 requant, second GEMM, bf16
  out) and a dense E=1, k=1 reduction against float64 torch ops.
- combine: identity experts with gates summing to one give y == x exactly;
  float64 weighted sum within half a bf16 ulp.
- the hand-worked two-token layer in tests/golden/worked_layer_t2.txt.
"""
import math
import os

import numpy as np
import pytest
import torch

from block_scaled_fp8_router_gb300 import synthetic as S
from tests.helpers import bf16_bits, bf16_to_f64, bits_to_bf16, e4m3_to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ dispatch

@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (37, 3, 5), (512, 8, 256), (1000, 6, 64)])
def test_dispatch_against_torch(oracle, T, k, E):
    g = torch.Generator().manual_seed(T + k + E)
    ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    counts, offsets, s2s, sl2, dropped = oracle.dispatch(ids.numpy(), E)
    assert dropped == 0
    flat = ids.flatten().long()
    np.testing.assert_array_equal(counts, torch.bincount(flat, minlength=E).numpy())
    assert counts.sum() == T * k
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    np.testing.assert_array_equal(s2s, torch.sort(flat, stable=True).indices.numpy())
    np.testing.assert_array_equal(sl2[s2s], np.arange(T * k))
    np.testing.assert_array_equal(s2s[sl2], np.arange(T * k))


def test_dispatch_brute_force_tiny(oracle):
    ids = np.array([[2, 0], [2, 1], [0, 2]], np.int32)
    counts, offsets, s2s, sl2, _ = oracle.dispatch(ids, 4)
    assert list(counts) == [2, 1, 3, 0]
    assert list(offsets) == [0, 2, 3, 6, 6]
    assert list(s2s) == [1, 4, 3, 0, 2, 5]
    assert list(sl2) == [3, 0, 4, 2, 1, 5]


def test_dispatch_drops_out_of_range(oracle):
    ids = np.array([[2, 9], [-1, 1], [0, 2]], np.int32)
    counts, offsets, s2s, sl2, dropped = oracle.dispatch(ids, 4)
    assert dropped == 2 and list(counts) == [1, 1, 2, 0] and offsets[-1] == 4
    assert sl2[1] == -1 and sl2[2] == -1
    assert list(s2s[:4]) == [4, 3, 0, 5] and np.all(s2s[4:] == -1)


def test_gather_rows(oracle):
    ids = np.array([[1, 0], [0, 1], [1, 1]], np.int32)
    _, offsets, s2s, _, _ = oracle.dispatch(ids, 2)
    rows = np.arange(3 * 5, dtype=np.uint16).reshape(3, 5)
    got = oracle.gather_rows(rows, s2s, int(offsets[-1]), 2)
    np.testing.assert_array_equal(got, rows[s2s // 2])


# ------------------------------------------------------------------ GEMM

def _dequant_rows(q, s):
    return e4m3_to_f64(q) * np.repeat(s.astype(np.float64), 128, axis=1)


def _dequant_blocks(q, s):
    return e4m3_to_f64(q) * np.repeat(np.repeat(s.astype(np.float64), 128, axis=0), 128, axis=1)


@pytest.mark.parametrize("M,N,K", [(3, 128, 128), (17, 256, 896), (5, 384, 2048)])
def test_fp8_gemm_against_float64(oracle, M, N, K):
    g = torch.Generator().manual_seed(M * N + K)
    a = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    aq, as_ = oracle.quant_1x128(bf16_bits(a))
    wq, ws = oracle.quant_128x128(bf16_bits(w))
    got = oracle.fp8_gemm(aq, as_, wq, ws).astype(np.float64)
    A, W = _dequant_rows(aq, as_), _dequant_blocks(wq, ws)
    ref = A @ W.T
    mag = np.abs(A) @ np.abs(W).T
    bound = (K // 128 + 3) * 2.0 ** -23 * mag
    assert np.all(np.abs(got - ref) <= bound)
    # a transposed or shifted operand would be far off
    assert np.abs(got - ref).max() < 1e-3 * np.abs(ref).max()


# ------------------------------------------------------------------ FFN

def _tiny_expert_setup(oracle, cfg, E_used, n_rows, seed=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n_rows, cfg.d, generator=g).to(torch.bfloat16)
    xq, xs = oracle.quant_1x128(bf16_bits(x))
    w13q, w13s, w2q, w2s = [], [], [], []
    for e in range(E_used):
        q, s = oracle.quant_128x128(bf16_bits(S.make_w13_expert(cfg, e, "cpu", seed)))
        w13q.append(q); w13s.append(s)
        q, s = oracle.quant_128x128(bf16_bits(S.make_w2_expert(cfg, e, "cpu", seed)))
        w2q.append(q); w2s.append(s)
    return xq, xs, np.stack(w13q), np.stack(w13s), np.stack(w2q), np.stack(w2s)


def test_ffn_composition(oracle):
    cfg = S.CONFIGS["tiny"]
    xq, xs, w13q, w13s, w2q, w2s = _tiny_expert_setup(oracle, cfg, 3, 9)
    row_e = np.array([0, 1, 2, 0, 1, 2, 2, 2, 0], np.int32)
    act_f, act_q, act_s, out = oracle.expert_ffn(xq, xs, row_e, w13q, w13s, w2q, w2s)
    F = cfg.F
    for r in range(len(row_e)):
        e = row_e[r]
        h = oracle.fp8_gemm(xq[r:r + 1], xs[r:r + 1], w13q[e], w13s[e])[0].astype(np.float64)
        g_, u = h[:F], h[F:]
        act = (g_ / (1.0 + np.exp(-g_)) * u).astype(np.float32)
        np.testing.assert_array_equal(act_f[r], act)
        o = oracle.fp8_gemm(act_q[r:r + 1], act_s[r:r + 1], w2q[e], w2s[e])[0]
        np.testing.assert_array_equal(out[r], bf16_bits(torch.from_numpy(o).to(torch.bfloat16)))
    # the requantised act obeys the block-quantiser invariants
    dq = e4m3_to_f64(act_q).reshape(-1, 128)
    assert np.all(np.abs(dq).max(axis=1) == 448.0)
    act_blocks = act_f.astype(np.float64).reshape(-1, 128)
    sc = act_s.reshape(-1).astype(np.float64)
    np.testing.assert_array_equal(sc, (np.abs(act_blocks).max(1).astype(np.float32) / np.float32(448)))
    ratio = np.abs(act_blocks / sc[:, None])
    top = np.maximum(ratio, np.abs(dq))
    spacing = np.where(top < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(top, 1e-30))) - 3))
    assert np.all(np.abs(act_blocks - dq * sc[:, None]) <= (spacing / 2 + 2.0 ** -23 * ratio) * sc[:, None] * (1 + 1e-12))


def test_ffn_dense_reduction_against_float64(oracle):
    """E = 1, k = 1: the layer is a dense SwiGLU FFN of the dequantised
    operands; compare with float64 torch ops (requant error dominates)."""
    cfg = S.CONFIGS["tiny"]
    xq, xs, w13q, w13s, w2q, w2s = _tiny_expert_setup(oracle, cfg, 1, 16, seed=4)
    row_e = np.zeros(16, np.int32)
    act_f, act_q, act_s, out = oracle.expert_ffn(xq, xs, row_e, w13q, w13s, w2q, w2s)
    X = torch.from_numpy(_dequant_rows(xq, xs))
    W13 = torch.from_numpy(_dequant_blocks(w13q[0], w13s[0]))
    W2 = torch.from_numpy(_dequant_blocks(w2q[0], w2s[0]))
    h = X @ W13.T
    act = torch.nn.functional.silu(h[:, :cfg.F]) * h[:, cfg.F:]
    np.testing.assert_allclose(act_f, act.numpy(), rtol=1e-5, atol=1e-5 * act.abs().max().item())
    y = act @ W2.T
    o = bf16_to_f64(out)
    err = np.abs(o - y.numpy()).max(axis=1) / np.abs(y.numpy()).max(axis=1)
    # the 1x128 requantisation of act (E4M3: up to 1/16 relative per element)
    # is the dominant difference from unquantised act; a few percent of the
    # row maximum is expected, a wrong operand gives O(1)
    assert err.max() < 8e-2
    # act_q @ W2 exactly (up to fp32 promotion) reproduces the bf16 output
    A = torch.from_numpy(_dequant_rows(act_q, act_s))
    y2 = (A @ W2.T).numpy()
    assert np.all(np.abs(o - y2) <= np.abs(y2) * 2.0 ** -8 + 1e-6 * np.abs(y2).max())


# ------------------------------------------------------------------ combine

def test_combine_identity_experts_exact(oracle):
    cfg = S.CONFIGS["long_dispatch"].with_(T=300, d=256)
    x = bf16_bits(S.make_x(cfg, "cpu"))
    ids = S.make_replay_payload(cfg, "cpu")[0].T.contiguous().numpy()
    gates = S.make_dirichlet_gates(cfg, "cpu").numpy()
    _, offsets, s2s, sl2, _ = oracle.dispatch(ids, cfg.E)
    rows = oracle.gather_rows(x, s2s, int(offsets[-1]), cfg.k)
    y = oracle.combine(rows, sl2, gates)
    np.testing.assert_array_equal(y, x)


def test_combine_against_float64(oracle):
    g = torch.Generator().manual_seed(2)
    T, k, d = 50, 4, 128
    out = torch.randn(T * k, d, generator=g).to(torch.bfloat16)
    gates = torch.rand(T, k, generator=g)
    sl2 = torch.randperm(T * k, generator=g).to(torch.int32)
    y = oracle.combine(bf16_bits(out), sl2.numpy(), gates.numpy())
    ref = (gates.double()[:, :, None] * out.double()[sl2.long()].view(T, k, d)).sum(1)
    yb = bits_to_bf16(y).double()
    ulp = 2.0 ** (torch.floor(torch.log2(ref.abs().clamp_min(1e-30))) - 7)
    assert torch.all((yb - ref).abs() <= 0.5 * ulp + 1e-5 * ref.abs())
    sl2_drop = sl2.clone()
    sl2_drop[::k] = -1                            # an unrouted slot contributes nothing
    y2 = bits_to_bf16(oracle.combine(bf16_bits(out), sl2_drop.numpy(), gates.numpy())).double()
    ref2 = ref - gates.double()[:, 0:1] * out.double()[sl2.long()[::k]]
    assert torch.allclose(y2, ref2, rtol=1e-2, atol=1e-2)


# ------------------------------------------------------------------ worked example

def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, *rest = line.split()
                vals[key] = rest
    return vals


def test_worked_layer_t2(oracle):
    gd = _golden("worked_layer_t2.txt")
    d = F = 128
    bf = lambda a: bf16_bits(torch.tensor(a, dtype=torch.float32).to(torch.bfloat16))
    x = bf([[0.875] * d, [-0.4375] * d])
    wr = bf([[0.0625] * d, [-0.0625] * d])
    w13 = [bf([[0.875] * d] * F + [[0.4375] * d] * F), bf([[-0.4375] * d] * F + [[0.875] * d] * F)]
    w2 = [bf([[0.21875] * F] * d), bf([[0.4375] * F] * d)]
    l = oracle.router_logits(x, wr)
    np.testing.assert_array_equal(l.reshape(-1), np.array(gd["logits"], np.float32))
    ids = oracle.topk(l, 1)
    np.testing.assert_array_equal(ids.reshape(-1), np.array(gd["ids"], np.int32))
    g = oracle.gates(l, ids, S.SOFTMAX, 1, 1.0)
    np.testing.assert_array_equal(g.reshape(-1), np.array(gd["gates"], np.float32))
    counts, offsets, s2s, sl2, _ = oracle.dispatch(ids, 2)
    np.testing.assert_array_equal(counts, np.array(gd["counts"], np.int32))
    np.testing.assert_array_equal(offsets, np.array(gd["offsets"], np.int32))
    xq, xs = oracle.quant_1x128(x)
    np.testing.assert_array_equal(xs.reshape(-1), np.array(gd["x_scales"], np.float32))
    assert np.all(xq[0] == int(gd["x_code_row0"][0], 16)) and np.all(xq[1] == int(gd["x_code_row1"][0], 16))
    wq = [oracle.quant_128x128(w) for w in w13]
    w2q = [oracle.quant_128x128(w) for w in w2]
    xq_s = oracle.gather_rows(xq, s2s, 2, 1)
    xs_s = oracle.gather_rows(xs, s2s, 2, 1)
    row_e = np.array([e for e in range(2) for _ in range(counts[e])], np.int32)
    act_f, act_q, act_s, out = oracle.expert_ffn(
        xq_s, xs_s, row_e, np.stack([q for q, _ in wq]), np.stack([s for _, s in wq]),
        np.stack([q for q, _ in w2q]), np.stack([s for _, s in w2q]))
    np.testing.assert_array_equal(act_f[:, 0], np.array(gd["act"], np.float32))
    assert np.all(act_f == act_f[:, :1])
    np.testing.assert_array_equal(act_s.reshape(-1), np.array(gd["act_scales"], np.float32))
    assert np.all(act_q[0] == int(gd["act_code_row0"][0], 16)) and np.all(act_q[1] == int(gd["act_code_row1"][0], 16))
    y = oracle.combine(out, sl2, g)
    yf = bf16_to_f64(y)
    np.testing.assert_array_equal(yf[:, 0], np.array(gd["y"], np.float64))
    assert np.all(yf == yf[:, :1])
