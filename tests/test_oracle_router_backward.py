"""Pins for the oracle's router backward (fixed ids, gradients through the
gates into the logits, the router weights and the tokens).

- float64 torch autograd of the router as a program: logits = x W_r^T in
  float64, the chosen logits gathered, the gate function (softmax or sigmoid,
  renormalised or not, times route_scale), loss = sum(gates * d_gates); the
  oracle's d_logits, dx and dW_r against its gradients.  The oracle's logits
  are the binary32 fma chain, so the comparison allows for their rounding.
- closed forms: with renormalisation a constant upstream gradient (and k = 1)
  gives zero; softmax logit gradients of a token sum to zero; an expert no
  token chose has a zero dW_r row; invalid tokens contribute nothing.
- a hand-worked three-token case (tests/golden/worked_router_backward.txt):
  exact values in all three gate modes.
"""
import numpy as np
import pytest
import torch

from tests.helpers import bf16_bits, bf16_to_f64


def _case(T, d, E, k, seed, w_std=0.02):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, d), generator=g).to(torch.bfloat16)
    wr = (torch.randn((E, d), generator=g) * w_std).to(torch.bfloat16)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    dg = torch.randn((T, k), generator=g)
    return x, wr, ids, dg


def _autograd(x, wr, ids, dg, score_fn, renorm, rs):
    x64 = torch.from_numpy(bf16_to_f64(bf16_bits(x))).requires_grad_(True)
    w64 = torch.from_numpy(bf16_to_f64(bf16_bits(wr))).requires_grad_(True)
    logits = x64 @ w64.T
    sel = torch.gather(logits, 1, ids.long())
    sel.retain_grad()
    if score_fn == 0:
        gates = torch.softmax(sel, dim=1)
    else:
        s = torch.sigmoid(sel)
        gates = s / s.sum(1, keepdim=True) if renorm else s
    (gates * rs * dg.double()).sum().backward()
    return sel.grad.numpy(), x64.grad.numpy(), w64.grad.numpy()


def _close(got, ref, rel):
    scale = max(np.abs(ref).max(), 1e-30)
    assert np.abs(got - ref).max() <= rel * scale, (np.abs(got - ref).max(), scale)


@pytest.mark.parametrize("score_fn,renorm,rs,k", [(0, 1, 1.0, 6), (1, 1, 1.0, 8), (1, 0, 2.5, 8), (1, 1, 2.5, 3),
                                                  (0, 1, 0.5, 2)])
def test_against_float64_autograd(oracle, score_fn, renorm, rs, k):
    x, wr, ids, dg = _case(96, 256, 24, k, seed=10 * k + score_fn)
    dl, dx, dw = oracle.router_backward(bf16_bits(x), bf16_bits(wr), ids.numpy(), dg.numpy(), score_fn, renorm, rs)
    rdl, rdx, rdw = _autograd(x, wr, ids, dg, score_fn, renorm, rs)
    _close(dl, rdl, 1e-5)
    _close(dx, rdx, 1e-5)
    _close(dw, rdw, 1e-5)


def test_constant_upstream_gradient_and_single_expert_give_zero(oracle):
    """With renormalisation the gates sum to route_scale whatever the logits,
    so a constant d_gates (and any d_gates when k = 1) moves nothing."""
    for score_fn in (0, 1):
        x, wr, ids, _ = _case(40, 128, 16, 5, seed=3)
        dg = np.full((40, 5), 0.75, np.float32)
        dl, dx, dw = oracle.router_backward(bf16_bits(x), bf16_bits(wr), ids.numpy(), dg, score_fn, 1, 2.0)
        assert np.abs(dl).max() <= 1e-12 and np.abs(dx).max() <= 1e-10 and np.abs(dw).max() <= 1e-10
        x, wr, ids, dg = _case(40, 128, 16, 1, seed=4)
        dl, dx, dw = oracle.router_backward(bf16_bits(x), bf16_bits(wr), ids.numpy(), dg.numpy(), score_fn, 1, 1.0)
        assert np.abs(dl).max() <= 1e-12


def test_softmax_gradients_sum_to_zero(oracle):
    x, wr, ids, dg = _case(64, 128, 32, 7, seed=5)
    dl, _, _ = oracle.router_backward(bf16_bits(x), bf16_bits(wr), ids.numpy(), dg.numpy(), 0, 1, 1.0,
                                      want_dx=False, want_dw=False)
    assert np.all(np.abs(dl.astype(np.float64).sum(1)) <= 1e-6 * np.abs(dl).sum(1) + 1e-12)


def test_unchosen_experts_and_invalid_tokens(oracle):
    x, wr, ids, dg = _case(50, 128, 12, 4, seed=6)
    ids = ids.numpy() % 10                               # experts 10, 11 never chosen ...
    ids[:, 1:] = (ids[:, :1] + np.arange(1, 4)) % 10     # ... and each token's ids distinct
    valid = np.ones(50, np.uint8)
    valid[7] = valid[30] = 0
    dl, dx, dw = oracle.router_backward(bf16_bits(x), bf16_bits(wr), ids, dg.numpy(), 1, 1, 1.0, valid=valid)
    assert np.all(dw[10:] == 0) and np.all(dl[[7, 30]] == 0) and np.all(dx[[7, 30]] == 0)
    # the invalid tokens are left out of dW_r: zeroing their upstream gradient changes nothing
    dg2 = dg.numpy().copy()
    dg2[[7, 30]] = 0
    _, _, dw2 = oracle.router_backward(bf16_bits(x), bf16_bits(wr), ids, dg2, 1, 1, 1.0, valid=valid)
    np.testing.assert_array_equal(dw, dw2)


def test_worked_router_backward(oracle):
    """The hand-worked three-token case in tests/golden/worked_router_backward.txt
    (every chosen logit exactly zero, so every gradient is a short binary
    fraction derived in the file's comments), in all three gate modes."""
    import os
    gd = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "worked_router_backward.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, *rest = line.split()
                gd[key] = [float(v) for v in rest]
    bf = lambda a, shape: bf16_bits(torch.tensor(a, dtype=torch.float32).reshape(shape).to(torch.bfloat16))
    x, wr = bf(gd["x"], (3, 2)), bf(gd["w_r"], (4, 2))
    ids = np.array(gd["ids"], np.int32).reshape(3, 2)
    dg = np.array(gd["d_gates"], np.float32).reshape(3, 2)
    np.testing.assert_array_equal(oracle.router_logits(x, wr)[:, :3], np.zeros((3, 3), np.float32))
    for mode in "ABC":
        score_fn, renorm, rs = gd[f"{mode}_mode"]
        dl, dx, dw = oracle.router_backward(x, wr, ids, dg, int(score_fn), int(renorm), rs)
        np.testing.assert_array_equal(dl.reshape(-1), np.array(gd[f"{mode}_d_logits"], np.float32), err_msg=mode)
        np.testing.assert_array_equal(dx.reshape(-1), np.array(gd[f"{mode}_dx"], np.float32), err_msg=mode)
        np.testing.assert_array_equal(dw.reshape(-1), np.array(gd[f"{mode}_dw"], np.float32), err_msg=mode)
