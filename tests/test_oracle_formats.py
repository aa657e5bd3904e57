"""Pins for the oracle's scalar formats (bf16 rounding, E4M3 encode/decode).

Checked against things other than the oracle itself: the OFP8 anchor table
(tests/golden/e4m3_ofp8_anchors.txt), torch's float8_e4m3fn and bfloat16
casts (library round-to-nearest-even), and exhaustive midpoint enumeration.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_e4m3_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def test_e4m3_anchor_table(oracle):
    with open(os.path.join(GOLDEN, "e4m3_ofp8_anchors.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) >= 8
    for code, val in rows:
        c = int(code, 16)
        got = oracle.e4m3_decode(c)
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code
            assert oracle.e4m3_encode(float(val)) == c


def test_e4m3_decode_matches_torch_all_codes(oracle):
    ref = _torch_e4m3_values()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got)
        else:
            assert got == ref[c], hex(c)


def test_e4m3_roundtrip_every_finite_code(oracle):
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_e4m3_midpoints_round_to_even(oracle):
    """Every midpoint between adjacent positive codes goes to the even code;
    one float32 ulp either side goes to the nearer neighbour."""
    for c in range(0, 0x7E):
        a, b = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = np.float32((a + b) / 2)           # <= 5 significant bits: exact
        assert float(mid) == (a + b) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(float(mid)) == even, hex(c)
        assert oracle.e4m3_encode(float(mid)) | 0x80 == oracle.e4m3_encode(float(-mid))
        lo = np.nextafter(mid, np.float32(0))
        hi = np.nextafter(mid, np.float32(np.inf))
        assert oracle.e4m3_encode(float(lo)) == c
        assert oracle.e4m3_encode(float(hi)) == c + 1


def test_e4m3_saturates(oracle):
    for v in [448.0, 463.99, 464.0, 479.0, 480.0, 1e6, 3.0e38, float(np.finfo(np.float32).max)]:
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE


def test_e4m3_zero_and_tiny(oracle):
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00          # tie between 0 and 2^-9 -> even (0)
    assert oracle.e4m3_encode(np.nextafter(np.float32(2.0 ** -10), np.float32(1))) == 0x01
    assert oracle.e4m3_encode(1e-30) == 0x00
    assert oracle.e4m3_encode(-1e-30) == 0x80
    assert oracle.e4m3_encode(float(np.float32(1e-45))) == 0x00  # denormal binary32


def test_e4m3_matches_torch_cast_random(oracle):
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 100,
        rng.uniform(-463.9, 463.9, 20000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-2).astype(np.float32),
        (rng.standard_normal(5000) * 1e-4).astype(np.float32),
    ])
    v = v[np.abs(v) < 464]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x)) for x in v], dtype=np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_bf16_rounding_matches_torch(oracle):
    rng = np.random.default_rng(1)
    f = rng.standard_normal(20000).astype(np.float32) * np.float32(3.7)
    # exact ties: low 16 bits == 0x8000
    bits = rng.integers(0, 2 ** 31, 2000, dtype=np.int64).astype(np.uint32)
    ties = ((bits & ~np.uint32(0xFFFF)) | np.uint32(0x8000)).view(np.float32)
    ties = ties[np.isfinite(ties)]
    vals = np.concatenate([f, ties, np.array([0.0, -0.0, 65504.0, 3.3895314e38], np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.uint16).numpy()
    got = np.array([oracle.f32_to_bf16(float(x)) for x in vals], dtype=np.uint16)
    np.testing.assert_array_equal(got, ref)
    for h in [0x0000, 0x8000, 0x3F80, 0xBF80, 0x7F7F, 0x0001]:
        assert oracle.bf16_to_f32(h) == torch.tensor([h], dtype=torch.int32).to(torch.int16).view(
            torch.bfloat16).float().item()
