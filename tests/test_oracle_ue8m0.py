"""Pins for the oracle's power-of-two (UE8M0) block scaling, the MXFP8-style
variant of the recipe that the hardware block-scaled MMA consumes.

- the exponent rule, by exact float64 arithmetic on the block's bf16
  values: scale 2^(e-127) is the smallest power of two with
  amax <= 448 * scale (checked both ways: large enough, and half of it is
  too small), at exact boundaries 448 * 2^p and their bf16 neighbours;
- codes: torch's float8_e4m3fn cast of v / scale (an exact division by a
  power of two), never saturating, block maximum in [224, 448];
- special blocks: zero, signed zero, tiny and huge magnitudes;
- the SwiGLU FFN with power-of-two scales on a dense E = 1 reduction
  against float64 torch ops on the dequantised operands.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_router_gb300 import synthetic as S
from tests.helpers import bf16_bits, bf16_to_f64, e4m3_to_f64


def _check_rule(v64, e):
    """v64 [nb, n] block values (exact), e [nb] biased exponents."""
    amax = np.abs(v64).max(axis=1)
    scale = np.ldexp(1.0, e.astype(np.int64) - 127)
    nz = amax > 0
    assert np.all(e[~nz] == 127)
    assert np.all(amax[nz] <= 448.0 * scale[nz])
    low = nz & (e > 0)                                      # e = 0: the clamp at 2^-127
    assert np.all(amax[low] > 448.0 * scale[low] / 2)      # minimal power of two


def _check_codes(v64, q, e):
    scale = np.ldexp(1.0, e.astype(np.int64) - 127)
    ratio = torch.from_numpy((v64 / scale[:, None]).astype(np.float32))   # exact: power-of-two division
    np.testing.assert_array_equal(q, ratio.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    dq = np.abs(e4m3_to_f64(q))
    nz = (np.abs(v64).max(axis=1) > 0) & (e > 0)           # e = 0: clamped, may sit lower
    assert np.all(dq.max(axis=1) <= 448.0)
    assert np.all(dq[nz].max(axis=1) >= 224.0)


@pytest.mark.parametrize("rows,cols,std", [(7, 256, 1.0), (33, 1024, 0.02), (5, 7168, 3.0)])
def test_ue8m0_1x128_random(oracle, rows, cols, std):
    g = torch.Generator().manual_seed(rows * cols)
    x = (torch.randn(rows, cols, generator=g) * std).to(torch.bfloat16)
    q, e = oracle.quant_ue8m0(bf16_bits(x), 1)
    assert q.shape == (rows, cols) and e.shape == (rows, cols // 128)
    v = bf16_to_f64(bf16_bits(x)).reshape(-1, 128)
    _check_rule(v, e.reshape(-1))
    _check_codes(v, q.reshape(-1, 128), e.reshape(-1))


def test_ue8m0_boundaries_and_special_blocks(oracle):
    rows = []
    for p in (-120, -9, -1, 0, 3, 100):
        base = 448.0 * 2.0 ** p
        for amax in (base, base * (1 + 2.0 ** -7), base * (1 - 2.0 ** -8)):   # bf16 neighbours of the boundary
            r = np.linspace(-amax / 3, amax / 5, 128)
            r[17] = -amax
            rows.append(r)
    rows.append(np.zeros(128))
    z = np.zeros(128)
    z[::2] = -0.0
    rows.append(z)
    rows.append(np.full(128, 2.0 ** -133))                 # bf16 subnormal
    x = torch.tensor(np.stack(rows), dtype=torch.float64).to(torch.bfloat16)
    v = bf16_to_f64(bf16_bits(x))
    q, e = oracle.quant_ue8m0(bf16_bits(x), 1)
    _check_rule(v, e[:, 0])
    _check_codes(v, q, e[:, 0])
    # exact boundary: the block maximum maps to 448 itself
    for i, p in enumerate((-120, -9, -1, 0, 3, 100)):
        assert e[3 * i, 0] == p + 127 and e[3 * i + 1, 0] == p + 128 and e[3 * i + 2, 0] == p + 127
        assert e4m3_to_f64(q[3 * i, 17]) == -448.0
    assert e[-3, 0] == 127 and np.all(q[-3] == 0)
    assert np.all(q[-2, ::2] == 0x80) and np.all(q[-2, 1::2] == 0)
    assert e[-1, 0] == 0                                    # 2^-133 needs 2^-135: clamped to 2^-127


def test_ue8m0_128x128(oracle):
    g = torch.Generator().manual_seed(5)
    w = (torch.randn(256, 384, generator=g) * 0.006).to(torch.bfloat16)
    w[:128, 128:256] = 0
    q, e = oracle.quant_ue8m0(bf16_bits(w), 128)
    assert e.shape == (2, 3)
    v = bf16_to_f64(bf16_bits(w))
    blocks = v.reshape(2, 128, 3, 128).transpose(0, 2, 1, 3).reshape(6, -1)
    qb = q.reshape(2, 128, 3, 128).transpose(0, 2, 1, 3).reshape(6, -1)
    _check_rule(blocks, e.reshape(-1))
    _check_codes(blocks, qb, e.reshape(-1))
    assert e[0, 1] == 127


def _deq_rows(q, e):
    return e4m3_to_f64(q) * np.repeat(np.ldexp(1.0, e.astype(np.int64) - 127), 128, axis=1)


def _deq_blocks(q, e):
    s = np.ldexp(1.0, e.astype(np.int64) - 127)
    return e4m3_to_f64(q) * np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)


def test_ue8m0_ffn_dense_reduction_against_float64(oracle):
    """E = 1: the SwiGLU FFN with power-of-two scales (act re-quantised by
    the same rule) against float64 torch ops on the dequantised operands."""
    cfg = S.CONFIGS["tiny"]
    g = torch.Generator().manual_seed(9)
    x = torch.randn(16, cfg.d, generator=g).to(torch.bfloat16)
    xq, xe = oracle.quant_ue8m0(bf16_bits(x), 1)
    w13q, w13e = oracle.quant_ue8m0(bf16_bits(S.make_w13_expert(cfg, 0, "cpu", 9)), 128)
    w2q, w2e = oracle.quant_ue8m0(bf16_bits(S.make_w2_expert(cfg, 0, "cpu", 9)), 128)
    f = oracle.ue8m0_value
    act_f, act_q, act_s, out = oracle.expert_ffn(xq, f(xe), np.zeros(16, np.int32), w13q[None], f(w13e)[None],
                                                 w2q[None], f(w2e)[None], ue8m0=True)
    # act scales are powers of two obeying the rule
    ea = (np.log2(act_s.astype(np.float64)) + 127).astype(np.int64)
    assert np.all(np.ldexp(1.0, ea - 127) == act_s)
    _check_rule(act_f.astype(np.float64).reshape(-1, 128), ea.reshape(-1))
    X = torch.from_numpy(_deq_rows(xq, xe))
    W13 = torch.from_numpy(_deq_blocks(w13q, w13e))
    W2 = torch.from_numpy(_deq_blocks(w2q, w2e))
    h = X @ W13.T
    act = torch.nn.functional.silu(h[:, :cfg.F]) * h[:, cfg.F:]
    np.testing.assert_allclose(act_f, act.numpy(), rtol=1e-5, atol=1e-5 * act.abs().max().item())
    A = torch.from_numpy(e4m3_to_f64(act_q) * np.repeat(act_s.astype(np.float64), 128, axis=1))
    y2 = (A @ W2.T).numpy()
    o = bf16_to_f64(out)
    assert np.all(np.abs(o - y2) <= np.abs(y2) * 2.0 ** -8 + 1e-6 * np.abs(y2).max())
