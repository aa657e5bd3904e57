"""Pins for the oracle's router: logits, top-k, gates, replay.

- logits: an exact-rational simulation of the binary32 fma chain (Python
  Fractions, correct rounding written out in integers) on small d; exact
  integer dot products when all partial sums are representable; float64
  matmul agreement (catches a transposed or misindexed operand).
- top-k: brute force over all subsets for small E; torch.topk on tie-free
  data; crafted ties, signed zeros and NaN.
- gates: torch softmax / sigmoid in float64; closed forms (k = 1, sums).
- replay: exact copy of the payload slab; capture -> replay round trip;
  invalid ids flagged.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest
import torch

from block_scaled_fp8_router_gb300 import synthetic as S
from tests.helpers import bf16_bits, bf16_to_f64


def _round_f32(q: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 (ties to even), with
    subnormals; overflow is not exercised here."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    # a in [2^e, 2^(e+1)); quantum 2^(e-23), or 2^-149 in the subnormal range
    qexp = max(e - 23, -149)
    n = a / Fraction(2) ** qexp
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * Fraction(2) ** qexp


def _fma_chain_exact(x, w):
    acc = Fraction(0)
    for a, b in zip(x, w):
        acc = _round_f32(Fraction(float(a)) * Fraction(float(b)) + acc)
    return float(acc)


def test_round_f32_helper_agrees_with_numpy():
    rng = np.random.default_rng(0)
    for v in rng.standard_normal(500) * 10.0 ** rng.integers(-40, 30, 500):
        assert float(_round_f32(Fraction(float(v)))) == float(np.float32(v))


@pytest.mark.parametrize("d", [1, 3, 8, 16])
def test_logits_fma_chain_exact_simulation(oracle, d):
    g = torch.Generator().manual_seed(d)
    x = torch.randn(5, d, generator=g).to(torch.bfloat16)
    w = (torch.randn(4, d, generator=g) * 0.37).to(torch.bfloat16)
    w[0, :] = torch.tensor([1e-38] * d).to(torch.bfloat16)    # products underflow into subnormals
    xb, wb = bf16_bits(x), bf16_bits(w)
    got = oracle.router_logits(xb, wb)
    xf, wf = bf16_to_f64(xb), bf16_to_f64(wb)
    for t in range(5):
        for e in range(4):
            assert got[t, e] == np.float32(_fma_chain_exact(xf[t], wf[e])), (t, e)


def test_logits_exact_on_integers(oracle):
    """Small integers: every partial sum is exact, so the chain equals the
    integer dot product."""
    rng = np.random.default_rng(3)
    xi = rng.integers(-8, 9, (9, 700))
    wi = rng.integers(-8, 9, (6, 700))
    xb = bf16_bits(torch.from_numpy(xi).to(torch.bfloat16))
    wb = bf16_bits(torch.from_numpy(wi).to(torch.bfloat16))
    got = oracle.router_logits(xb, wb)
    np.testing.assert_array_equal(got, (xi @ wi.T).astype(np.float32))


def test_logits_close_to_float64_matmul(oracle):
    cfg = S.CONFIGS["tiny"]
    x = S.make_x(cfg, "cpu")[:40]
    w = S.make_router_w(cfg, "cpu")
    got = oracle.router_logits(bf16_bits(x), bf16_bits(w))
    ref = x.double() @ w.double().T
    bound = (x.double().abs() @ w.double().abs().T) * cfg.d * 2.0 ** -24
    assert torch.all((torch.from_numpy(got).double() - ref).abs() <= bound)


def _brute_topk(l, k):
    """All k-subsets; the chosen set is the one no outside expert ranks
    before; slot order by rank.  Rank key: (is_nan, -value, index)."""
    E = len(l)
    key = lambda e: (np.isnan(l[e]), 0.0 if np.isnan(l[e]) else -float(l[e]), e)
    for sub in itertools.combinations(range(E), k):
        inside = set(sub)
        if all(key(i) < key(o) for i in inside for o in range(E) if o not in inside):
            return sorted(sub, key=key)
    raise AssertionError


@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (8, 3), (8, 8), (7, 4)])
def test_topk_brute_force(oracle, E, k):
    rng = np.random.default_rng(E * 10 + k)
    l = rng.integers(-3, 4, (300, E)).astype(np.float32)      # many ties
    l[::7] = rng.standard_normal((len(l[::7]), E)).astype(np.float32)
    l[3, :] = np.float32(np.nan)
    l[5, 1] = np.float32(np.nan)
    l[6, :2] = [0.0, -0.0]
    l[9, :] = -np.inf
    got = oracle.topk(l, k)
    for t in range(l.shape[0]):
        assert list(got[t]) == _brute_topk(l[t], k), t


def test_topk_matches_torch_on_tie_free(oracle):
    g = torch.Generator().manual_seed(11)
    l = torch.randn(500, 256, generator=g)
    got = oracle.topk(l.numpy(), 8)
    ref = torch.topk(l, 8, dim=1, largest=True, sorted=True).indices.numpy()
    np.testing.assert_array_equal(got, ref)


def test_topk_ties_and_signed_zero(oracle):
    l = np.zeros((3, 6), np.float32)
    l[1] = [-0.0, 0.0, -0.0, 0.0, -1.0, 1.0]
    l[2] = [np.nan, np.nan, 5, np.nan, -np.inf, np.nan]
    got = oracle.topk(l, 3)
    assert list(got[0]) == [0, 1, 2]
    assert list(got[1]) == [5, 0, 1]         # -0 == +0 -> lower index first
    assert list(got[2]) == [2, 4, 0]         # NaN ranks below -inf


@pytest.mark.parametrize("score_fn", [S.SOFTMAX, S.SIGMOID])
@pytest.mark.parametrize("renorm", [0, 1])
def test_gates_against_torch(oracle, score_fn, renorm):
    g = torch.Generator().manual_seed(7 + score_fn)
    l = (torch.randn(200, 32, generator=g) * 3).float()
    ids = oracle.topk(l.numpy(), 4)
    got = oracle.gates(l.numpy(), ids, score_fn, renorm, route_scale=2.5)
    ld = l.double()
    if score_fn == S.SOFTMAX:
        p = torch.softmax(ld, dim=1)
    else:
        p = torch.sigmoid(ld)
    sel = torch.gather(p, 1, torch.from_numpy(ids).long())
    if renorm:
        sel = sel / sel.sum(dim=1, keepdim=True)
    ref = (sel * 2.5).float().numpy()
    np.testing.assert_allclose(got, ref, rtol=2e-7, atol=0)
    if renorm:
        np.testing.assert_allclose(got.astype(np.float64).sum(1), 2.5, rtol=1e-6)


def test_gates_k1_and_invalid(oracle):
    l = np.random.default_rng(0).standard_normal((10, 8)).astype(np.float32)
    ids = oracle.topk(l, 1)
    for fn in (S.SOFTMAX, S.SIGMOID):
        assert np.all(oracle.gates(l, ids, fn, 1, 1.0) == 1.0)
    valid = np.ones(10, np.uint8)
    valid[4] = 0
    g = oracle.gates(l, ids, S.SOFTMAX, 1, 1.0, valid=valid)
    assert g[4, 0] == 0.0 and g[3, 0] == 1.0


def test_replay_copies_payload_slab(oracle):
    cfg = S.CONFIGS["replay"].with_(T=512)
    payload = S.make_replay_payload(cfg, "cpu").numpy()   # [1, k, T]
    ids, valid, bad = oracle.replay(payload[0], cfg.E)
    assert bad == 0 and np.all(valid == 1)
    np.testing.assert_array_equal(ids, payload[0].T)


def test_capture_replay_round_trip(oracle):
    cfg = S.CONFIGS["tiny"]
    x = bf16_bits(S.make_x(cfg, "cpu"))
    w = bf16_bits(S.make_router_w(cfg, "cpu"))
    l = oracle.router_logits(x, w)
    ids = oracle.topk(l, cfg.k)
    gates = oracle.gates(l, ids, cfg.score_fn, 1, 1.0)
    capture = np.ascontiguousarray(ids.T)                   # one [k, T] layer slab
    rid, valid, bad = oracle.replay(capture, cfg.E)
    assert bad == 0
    np.testing.assert_array_equal(rid, ids)
    np.testing.assert_array_equal(oracle.gates(l, rid, cfg.score_fn, 1, 1.0), gates)


def test_replay_flags_bad_ids(oracle):
    p = np.array([[0, 3, 9, 1, -1], [1, 3, 2, 7, 2]], np.int32)   # k=2, T=5, E=8
    ids, valid, bad = oracle.replay(p, 8)
    assert list(valid) == [1, 0, 0, 1, 0] and bad == 3
    np.testing.assert_array_equal(ids, p.T)


def test_router_worked_example(oracle):
    x = np.array([[0.875] * 128, [-0.4375] * 128], np.float32)
    w = np.array([[0.0625] * 128, [-0.0625] * 128], np.float32)
    xb = bf16_bits(torch.from_numpy(x).to(torch.bfloat16))
    wb = bf16_bits(torch.from_numpy(w).to(torch.bfloat16))
    l = oracle.router_logits(xb, wb)
    np.testing.assert_array_equal(l, [[7.0, -7.0], [-3.5, 3.5]])
    ids = oracle.topk(l, 1)
    np.testing.assert_array_equal(ids[:, 0], [0, 1])
