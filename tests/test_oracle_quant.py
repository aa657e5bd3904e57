"""Pins for the oracle's block-scaled quantisers (1x128 and 128x128).

Pinned by invariants that any correct block quantiser obeys (the block's
largest magnitude maps to +-448; dequantisation error within half an E4M3
ulp plus one binary32 rounding, times the scale) and by torch's
float8_e4m3fn cast applied block by block.
"""
import numpy as np
import pytest
import torch

from block_scaled_fp8_router_gb300 import synthetic as S
from tests.helpers import bf16_bits, bf16_to_f64, e4m3_to_f64


def _spacing(v):
    """E4M3 grid spacing in the binade of |v| (subnormal spacing below 2^-6)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))


def _check_blocks(v, q, s, blocks):
    """v: [nb, n] values (f64), q: [nb, n] codes, s: [nb] scales."""
    dq = e4m3_to_f64(q)
    nz = np.abs(v).max(axis=1) > 0
    # the block maximum becomes +-448 exactly
    assert np.all(np.abs(dq[nz]).max(axis=1) == 448.0)
    assert np.all(s[~nz] == 1.0) and np.all(dq[~nz] == 0)
    # |v - q s| <= (ulp/2 + 2^-23 |v/s|) s
    ratio = v / s[:, None].astype(np.float64)
    bound = (_spacing(np.maximum(np.abs(ratio), np.abs(dq))) / 2 + 2.0 ** -23 * np.abs(ratio)) * s[:, None]
    err = np.abs(v - dq * s[:, None].astype(np.float64))
    assert np.all(err <= bound * (1 + 1e-12))
    # against torch: s = amax / 448 in float32, codes = float8 cast of (v / s)
    amax = torch.from_numpy(np.abs(v).max(axis=1).astype(np.float32))
    s_ref = amax / torch.tensor(448.0, dtype=torch.float32)
    s_ref[s_ref == 0] = 1.0
    np.testing.assert_array_equal(s, s_ref.numpy())
    q_ref = (torch.from_numpy(v.astype(np.float32)) / s_ref[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    np.testing.assert_array_equal(q, q_ref.numpy())


@pytest.mark.parametrize("rows,cols,std", [(7, 256, 1.0), (33, 1024, 0.02), (5, 7168, 3.0)])
def test_quant_1x128(oracle, rows, cols, std):
    g = torch.Generator().manual_seed(rows * cols)
    x = (torch.randn(rows, cols, generator=g) * std).to(torch.bfloat16)
    xb = bf16_bits(x)
    q, s = oracle.quant_1x128(xb)
    assert q.shape == (rows, cols) and s.shape == (rows, cols // 128)
    v = bf16_to_f64(xb).reshape(rows * cols // 128, 128)
    _check_blocks(v, q.reshape(-1, 128), s.reshape(-1), None)


def test_quant_1x128_special_blocks(oracle):
    x = torch.zeros(3, 384, dtype=torch.bfloat16)
    x[0, 128:256] = -0.0                 # a block of negative zeros
    x[1, :128] = torch.linspace(-5, 5, 128)
    x[1, 200] = 1e-40                    # subnormal in an otherwise zero block
    x[2, 256:] = 448.0 * 2.0 ** -9       # constant block with an exact scale
    xb = bf16_bits(x)
    q, s = oracle.quant_1x128(xb)
    assert s[0, 0] == 1.0 and np.all(q[0, :128] == 0x00)
    assert s[0, 1] == 1.0 and np.all(q[0, 128:256] == 0x80)   # -0 keeps its sign
    assert s[2, 2] == 2.0 ** -9 and np.all(q[2, 256:] == 0x7E)
    assert q[1, 0] == 0xFE and q[1, 127] == 0x7E
    assert s[1, 1] == np.float32(np.float32(bf16_to_f64(xb)[1, 200]) / np.float32(448.0))


@pytest.mark.parametrize("rows,cols,std", [(128, 256, 0.02), (384, 128, 0.006), (256, 512, 1.0)])
def test_quant_128x128(oracle, rows, cols, std):
    g = torch.Generator().manual_seed(rows + cols)
    w = (torch.randn(rows, cols, generator=g) * std).to(torch.bfloat16)
    wb = bf16_bits(w)
    q, s = oracle.quant_128x128(wb)
    assert s.shape == (rows // 128, cols // 128)
    v = bf16_to_f64(wb).reshape(rows // 128, 128, cols // 128, 128).transpose(0, 2, 1, 3).reshape(-1, 128 * 128)
    qb = q.reshape(rows // 128, 128, cols // 128, 128).transpose(0, 2, 1, 3).reshape(-1, 128 * 128)
    _check_blocks(v, qb, s.reshape(-1), None)


def test_quant_128x128_equals_1x128_on_uniform_rows(oracle):
    """A 128x128 block whose rows all have the same max magnitude gets the same
    scale and codes as each of its rows quantised 1x128."""
    g = torch.Generator().manual_seed(5)
    w = torch.randn(128, 256, generator=g).clamp(-2.5, 2.5).to(torch.bfloat16)
    w[:, 0] = 7.0
    w[:, 128] = -3.0
    wb = bf16_bits(w)
    q1, s1 = oracle.quant_1x128(wb)
    q2, s2 = oracle.quant_128x128(wb)
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s1, np.repeat(s2, 128, axis=0))


def test_quant_synthetic_weight_shape(oracle):
    cfg = S.CONFIGS["tiny"]
    w13 = S.make_w13_expert(cfg, 0, "cpu")
    q, s = oracle.quant_128x128(bf16_bits(w13))
    assert q.shape == (2 * cfg.F, cfg.d) and s.shape == (2 * cfg.F // 128, cfg.d // 128)
    assert np.all((q & 0x7F) != 0x7F)   # never NaN
