"""The quantisers divide each element by its block scale through the scale's
correctly rounded reciprocal y = RN(1/s): q0 = RN(v*y), then correction
steps q <- RN(q + RN(v - q*s) * y) with fused multiply-adds (Markstein's
theorem; J.-M. Muller et al., Handbook of Floating-Point Arithmetic, division
with an FMA).  These tests emulate that arithmetic exactly in numpy (float64
holds every product of two floats and every residual exactly; the last
rounding of a sum is done by two-sum and an explicit tie break) and compare it
with IEEE division v / s, the quotient the oracle takes:

- one step, every bf16 v with |v| <= amax, every bf16 amax whose scale
  s = RN(amax / 448) is on the fast path (2^-90 <= s): the quotient equals
  RN(v / s) wherever |v / s| >= 2^-12, and every E4M3 code equals the code of
  RN(v / s) -- exhaustive over the 1 x 128 quantiser's input domain;
- two steps on fp32 values (random, near E4M3 rounding midpoints, tiny).

A check that the emulation can fail: the uncorrected RN(v*y) must disagree
with IEEE division on a large share of the same pairs."""
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

F32 = np.float32


def _e4m3_codes(x):
    t = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _rn32_of_sum(a, b):
    """RN to float32 of the exact sum a + b of two float64 values."""
    s = a + b
    bb = s - a
    err = (a - (s - bb)) + (b - bb)                  # a + b = s + err exactly
    r = s.astype(F32)
    up = np.nextafter(r, F32(np.inf))
    dn = np.nextafter(r, F32(-np.inf))
    r64 = r.astype(np.float64)
    at_up = (s == (r64 + up.astype(np.float64)) / 2) & (err != 0)
    at_dn = (s == (r64 + dn.astype(np.float64)) / 2) & (err != 0)
    out = np.where(at_up & (err > 0), up, r)
    out = np.where(at_dn & (err < 0), dn, out)
    return out


def _step(v, s, y, q):
    """RN32(q + RN32(v - q*s) * y) with both fused operations exact."""
    d = v.astype(np.float64) - q.astype(np.float64) * s.astype(np.float64)   # exact (Sterbenz)
    r = d.astype(F32)
    return _rn32_of_sum(q.astype(np.float64), r.astype(np.float64) * y.astype(np.float64))


def reciprocal_division(v, s, steps):
    y = (F32(1.0) / s).astype(F32)
    q0 = (v * y).astype(F32)
    q = q0
    for _ in range(steps):
        q = _step(v, s, y, q)
    return np.copysign(q, v), q0


_BF16_POS = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(F32)


def _amax_range(lo_hi):
    lo, hi = lo_hi
    n = mism = code_mism = naive = 0
    for i in range(lo, hi):
        amax = _BF16_POS[i]
        s = F32(amax) / F32(448.0)
        if s < F32(2.0 ** -90):
            continue
        v = _BF16_POS[: i + 1]
        sv = np.full_like(v, s)
        ref = v / sv
        q, q0 = reciprocal_division(v, sv, 1)
        big = ref >= F32(2.0 ** -12)
        n += len(v)
        mism += int(((q != ref) & big).sum())
        code_mism += int((_e4m3_codes(q) != _e4m3_codes(ref)).sum())
        naive += int(((q0 != ref) & big).sum())
    return n, mism, code_mism, naive


def test_one_step_exact_on_every_bf16_pair():
    nb = len(_BF16_POS)
    cuts = np.linspace(0, nb, 65).astype(int)
    chunks = list(zip(cuts[:-1], cuts[1:]))
    workers = max(1, min(8, os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(workers) as pool:
        res = pool.map(_amax_range, chunks)
    n, mism, code_mism, naive = (sum(r[i] for r in res) for i in range(4))
    assert n > 5e8                                   # every fast-path pair
    assert mism == 0 and code_mism == 0
    assert naive > 1e7                               # the correction step is needed


@pytest.mark.parametrize("mode", ["uniform", "log", "midpoints"])
def test_two_steps_exact_on_fp32_values(mode):
    rng = np.random.default_rng(["uniform", "log", "midpoints"].index(mode))
    n = 3_000_000
    amax = (rng.uniform(1, 2, n) * 2.0 ** rng.integers(-80, 120, n)).astype(F32)
    if mode == "uniform":
        u = rng.uniform(-1, 1, n)
    elif mode == "log":
        u = np.where(rng.random(n) < 0.5, -1, 1) * 2.0 ** rng.uniform(-40, 0, n)
    else:
        # v / s within a few ulps of an E4M3 rounding midpoint (1 + (2m+1)/16) 2^e
        m = rng.integers(0, 8, n)
        e = rng.integers(-9, 9, n)
        u = np.minimum((1 + (2 * m + 1) / 16.0) * 2.0 ** e / 448.0 * (1 + rng.normal(0, 2e-7, n)), 1.0)
    v = (amax.astype(np.float64) * u).astype(F32)
    s = (amax / F32(448.0)).astype(F32)
    ref = v / s
    q, q0 = reciprocal_division(v, s, 2)
    big = np.abs(ref) >= F32(2.0 ** -12)
    assert int(((q != ref) & big).sum()) == 0
    assert int((_e4m3_codes(q) != _e4m3_codes(ref)).sum()) == 0
    assert np.all(np.signbit(q[v == 0]) == np.signbit(v[v == 0]))
    assert int(((q0 != ref) & big).sum()) > n // 20


def _scale_binade(e):
    bits = (np.uint32(e + 127) << np.uint32(23)) | np.arange(1 << 23, dtype=np.uint32)
    a = bits.view(F32)
    q, _ = reciprocal_division(a, np.full_like(a, F32(448.0)), 1)
    return int((q.view(np.uint32) != (a / F32(448.0)).view(np.uint32)).sum())


def test_block_scale_one_step_on_every_binary32_amax():
    """amax / 448 from the constant RN(1/448) and one correction step equals
    IEEE division for every binary32 amax in [2^-100, 2^128)."""
    workers = max(1, min(8, os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(workers) as pool:
        bad = pool.map(_scale_binade, range(-100, 128))
    assert sum(bad) == 0


def test_emulated_fma_step_matches_exact_rationals():
    """The two-sum rounding against Python's exact fractions on a sample."""
    from fractions import Fraction
    rng = np.random.default_rng(7)
    v = rng.uniform(-1e3, 1e3, 2000).astype(F32)
    s = rng.uniform(1e-3, 10, 2000).astype(F32)
    y = (F32(1.0) / s).astype(F32)
    q = (v * y).astype(F32)
    got = _step(v, s, y, q)
    for i in range(len(v)):
        r = F32(Fraction(float(v[i])) - Fraction(float(q[i])) * Fraction(float(s[i])))
        exact = Fraction(float(q[i])) + Fraction(float(r)) * Fraction(float(y[i]))
        # RN32 of an exact rational: nearest of the two float32 neighbours
        lo = F32(float(exact))
        cand = [lo, np.nextafter(lo, F32(-np.inf)), np.nextafter(lo, F32(np.inf))]
        dist = [abs(Fraction(float(c)) - exact) for c in cand]
        best = min(dist)
        ties = [c for c, dd in zip(cand, dist) if dd == best]
        want = ties[0] if len(ties) == 1 else [c for c in ties if (c.view(np.uint32) & 1) == 0][0]
        assert got[i] == want, (i, v[i], s[i])


def _step_negated(v, s, y, q):
    """The scalar device form: RN32(q + (-RN32(q*s - v)) * y)."""
    d = q.astype(np.float64) * s.astype(np.float64) - v.astype(np.float64)   # exact
    r = d.astype(F32)
    return _rn32_of_sum(q.astype(np.float64), (-r).astype(np.float64) * y.astype(np.float64))


@pytest.mark.parametrize("steps", [1, 2])
def test_negated_residual_form_equals_copysign_form(steps):
    """The device takes the residual negated, RN(q*s - v), so that a zero
    dividend keeps its sign; the emulation above takes RN(v - q*s) and
    restores the sign of v at the end.  Both give the same bits for every
    value, zeros of both signs included, so the exhaustive checks above hold
    for the device's form."""
    rng = np.random.default_rng(steps)
    n = 1_000_000
    amax = (rng.uniform(1, 2, n) * 2.0 ** rng.integers(-80, 120, n)).astype(F32)
    v = (amax.astype(np.float64) * rng.uniform(-1, 1, n)).astype(F32)
    v[:1000] = F32(0.0)
    v[1000:2000] = F32(-0.0)
    v[2000:3000] = (amax[2000:3000] * F32(2.0 ** -30)).astype(F32)     # tiny quotients
    s = (amax / F32(448.0)).astype(F32)
    y = (F32(1.0) / s).astype(F32)
    qn = (v * y).astype(F32)
    for _ in range(steps):
        qn = _step_negated(v, s, y, qn)
    qc, _ = reciprocal_division(v, s, steps)
    assert np.array_equal(qn.view(np.uint32), qc.view(np.uint32))
    assert np.all(np.signbit(qn[:2000]) == np.signbit(v[:2000]))
