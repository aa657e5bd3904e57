"""Pins of the oracle's NVFP4 mode (the FP4 variant the prime-rl post lists as
future work, "RL at 1T Scale", closing section; NVIDIA's NVFP4 format as the
plainest reading): FP4 E2M1 values against the OCP Microscaling table, the
E2M1 rounding against a brute-force nearest-value search, the E4M3 block
scales against torch's e4m3 cast, quantisation error bounds, and the NVFP4
GEMM against a float64 product of operands decoded here."""
import os

import numpy as np
import pytest
import torch

from tests.helpers import bf16_bits, e4m3_to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_ocp_values.txt")


@pytest.fixture(scope="module")
def oracle():
    from oracle import oracle as O
    return O


def _ocp_table():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        c, v = line.split()
        vals[int(c, 16)] = float(v)
    assert len(vals) == 16
    return vals


def _decode_codes(codes: np.ndarray) -> np.ndarray:
    tab = _ocp_table()
    lut = np.array([tab[c] for c in range(16)], np.float64)
    return lut[codes]


def _unpack(q: np.ndarray) -> np.ndarray:
    """[rows, cols/2] packed -> [rows, cols] codes (element 2i low nibble)."""
    out = np.empty((q.shape[0], q.shape[1] * 2), np.uint8)
    out[:, 0::2] = q & 15
    out[:, 1::2] = q >> 4
    return out


def _brute_e2m1(v: float) -> int:
    """Nearest E2M1 value by exhaustive search over the OCP table, ties to the
    even code, magnitudes beyond 6 to 6; the sign of v is kept."""
    tab = _ocp_table()
    neg = np.signbit(np.float32(v))
    a = abs(float(v))
    best = None
    for c in range(8):
        d = abs(a - tab[c])
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    c = best[1] if a <= 6.0 else 7
    return c | (8 if neg else 0)


def test_e2m1_decode_matches_ocp_table(oracle):
    tab = _ocp_table()
    for c in range(16):
        got = oracle.e2m1_decode(c)
        assert got == tab[c] and np.signbit(got) == np.signbit(tab[c]), (c, got, tab[c])


def test_e2m1_encode_against_brute_force(oracle):
    g = np.random.default_rng(3)
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    mids = [(a + b) / 2 for a, b in zip(grid, grid[1:])] + [7.0]
    vals = list(g.uniform(-8, 8, 4000).astype(np.float32))
    for m in mids:
        for x in (m, np.nextafter(np.float32(m), np.float32(0)), np.nextafter(np.float32(m), np.float32(10))):
            vals += [np.float32(x), -np.float32(x)]
    vals += [np.float32(v) for v in (0.0, -0.0, 6.0, 6.5, 1e30, -1e30, 1e-30, -1e-30, 0.2499999, 5.999)]
    for v in vals:
        assert oracle.e2m1_encode(float(v)) == _brute_e2m1(v), v


def _nvfp4_input(g: torch.Generator, rows: int, cols: int) -> torch.Tensor:
    # block magnitudes spread over 2^-10 .. 2^6, an all-zero block, a block
    # with one large entry
    x = torch.randn(rows, cols, generator=g) * torch.exp2(torch.randint(-10, 6, (rows, cols // 16), generator=g)
                                                          .float()).repeat_interleave(16, dim=1)
    x[1, 16:32] = 0.0
    x[2, 32:48] = 1e-3
    x[2, 40] = 37.0
    return x.to(torch.bfloat16)


def test_quant_nvfp4_scales_codes_and_error(oracle):
    g = torch.Generator().manual_seed(5)
    rows, cols = 24, 256
    xb = _nvfp4_input(g, rows, cols)
    x = xb.float()
    q, s, s_enc = oracle.quant_nvfp4(bf16_bits(xb))
    assert q.shape == (rows, cols // 2) and s.shape == (rows, cols // 16)
    amax_t = x.abs().max()
    assert s_enc == (torch.tensor(6.0 * 448.0) / amax_t).item()
    # block scales: torch's e4m3 cast of (amax_block / 6) * s_enc in float32
    blocks = x.view(rows, cols // 16, 16)
    bd = (blocks.abs().amax(2) / torch.tensor(6.0)) * torch.tensor(s_enc)
    sref = bd.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(s, sref)
    assert s[1, 1] == 0 and np.all(_unpack(q)[1, 16:32] == 0)          # the all-zero block
    # codes: the brute-force rounding of x * (s_enc / scale) in float32
    sv = torch.from_numpy(e4m3_to_f64(s)).float()
    s_elem = torch.where(sv == 0, torch.zeros_like(sv), torch.tensor(s_enc) / sv)
    scaled = (blocks * s_elem[:, :, None]).reshape(rows, cols).numpy()
    codes = _unpack(q)
    for r in range(rows):
        for c in range(cols):
            assert codes[r, c] == _brute_e2m1(scaled[r, c]), (r, c, scaled[r, c])
    # error bound: within half the E2M1 spacing at the scaled magnitude, or
    # saturated at 6
    deq = _decode_codes(codes)
    a = np.abs(scaled.astype(np.float64))
    half = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))
    assert np.all(np.abs(deq - scaled) <= np.maximum(half, a - 6.0) + 1e-12)
    # a block's largest element scales to 6 times (unrounded scale / stored
    # scale): at most half an e4m3 step above 6 for normal scales, more when
    # the scale falls into the e4m3 subnormals (the format's range limit)
    nz = s != 0
    ratio = bd.double().numpy() / np.where(nz, e4m3_to_f64(s), 1.0)
    amax_scaled = a.reshape(rows, cols // 16, 16).max(2)
    assert np.all(np.abs(amax_scaled[nz] - 6.0 * ratio[nz]) <= 6.0 * ratio[nz] * 1e-6)
    normal = nz & (e4m3_to_f64(s) >= 2.0 ** -6)
    assert np.all(amax_scaled[normal] <= 6.0 * (1 + 2.0 ** -4) * (1 + 1e-6))


def test_gemm_nvfp4_against_float64(oracle):
    g = torch.Generator().manual_seed(9)
    M, N, K = 40, 24, 320
    a = (torch.randn(M, K, generator=g) * 3.0).to(torch.bfloat16)
    b = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    aq, as_, ae = oracle.quant_nvfp4(bf16_bits(a))
    bq, bs, be = oracle.quant_nvfp4(bf16_bits(b))
    out = oracle.gemm_nvfp4(aq, as_, ae, bq, bs, be)
    ad = _decode_codes(_unpack(aq)) * np.repeat(e4m3_to_f64(as_), 16, axis=1) / ae
    bd = _decode_codes(_unpack(bq)) * np.repeat(e4m3_to_f64(bs), 16, axis=1) / be
    ref = ad @ bd.T
    mag = np.abs(ad) @ np.abs(bd).T
    assert np.all(np.abs(out - ref) <= mag * 1e-13 + 1e-300)
    # and it approximates the unquantised product (4-bit operands: ~10% of
    # the typical entry)
    exact = a.double().numpy() @ b.double().numpy().T
    assert np.abs(out - exact).max() / np.abs(exact).max() < 0.25


def _deq(q, s, enc):
    return _decode_codes(_unpack(q)) * np.repeat(e4m3_to_f64(s), 16, axis=1) / enc


def test_expert_ffn_nvfp4_stages_against_float64(oracle):
    """Two experts (rows interleaved): GEMM1 against a float64 product of
    operands decoded here (within binary32 rounding), act against torch's
    float64 silu (within bf16 rounding), the act re-quantisation against the
    quantiser applied to that act, GEMM2 against float64 (within bf16
    rounding), and the whole FFN against the unquantised float64 SwiGLU
    layer (4-bit operands: a loose bound)."""
    from tests.helpers import bf16_to_f64
    g = torch.Generator().manual_seed(21)
    E, d, F, n = 2, 128, 96, 40
    x = torch.randn(n, d, generator=g).to(torch.bfloat16)
    w13 = (torch.randn(E, 2 * F, d, generator=g) * 0.05).to(torch.bfloat16)
    w2 = (torch.randn(E, d, F, generator=g) * 0.05).to(torch.bfloat16)
    re = (np.arange(n) % E).astype(np.int32)
    xq, xs, xe = oracle.quant_nvfp4(bf16_bits(x))
    qs = [oracle.quant_nvfp4(bf16_bits(w13[e])) for e in range(E)]
    q2 = [oracle.quant_nvfp4(bf16_bits(w2[e])) for e in range(E)]
    w13q, w13s = np.stack([a[0] for a in qs]), np.stack([a[1] for a in qs])
    w13e = np.array([a[2] for a in qs], np.float32)
    w2q, w2s = np.stack([a[0] for a in q2]), np.stack([a[1] for a in q2])
    w2e = np.array([a[2] for a in q2], np.float32)
    h, act, aq, as_, ae, out = oracle.expert_ffn_nvfp4(xq, xs, xe, re, w13q, w13s, w13e, w2q, w2s, w2e)
    xd = _deq(xq, xs, xe)
    h_ref = np.stack([xd[r] @ _deq(w13q[re[r]], w13s[re[r]], w13e[re[r]]).T for r in range(n)])
    assert np.all(np.abs(h - h_ref) <= np.abs(h_ref) * 2.0 ** -23 + 1e-30)
    gt, up = torch.from_numpy(h[:, :F]).double(), torch.from_numpy(h[:, F:]).double()
    act_ref = (torch.nn.functional.silu(gt) * up).numpy()
    assert np.all(np.abs(bf16_to_f64(act) - act_ref) <= np.abs(act_ref) * 2.0 ** -8 + 1e-30)
    rq, rs, renc = oracle.quant_nvfp4(act)
    np.testing.assert_array_equal(aq, rq)
    np.testing.assert_array_equal(as_, rs)
    assert ae == renc
    ad = _deq(aq, as_, ae)
    out_ref = np.stack([ad[r] @ _deq(w2q[re[r]], w2s[re[r]], w2e[re[r]]).T for r in range(n)])
    assert np.all(np.abs(bf16_to_f64(out) - out_ref) <= np.abs(out_ref) * 2.0 ** -8 * (1 + 2.0 ** -20) + 1e-30)
    # end to end against the unquantised layer
    xf = x.double()
    exact = []
    for r in range(n):
        hh = xf[r] @ w13[re[r]].double().T
        a = torch.nn.functional.silu(hh[:F]) * hh[F:]
        exact.append((a @ w2[re[r]].double().T).numpy())
    exact = np.stack(exact)
    err = np.abs(bf16_to_f64(out) - exact).max(1) / np.abs(exact).max(1)
    assert err.max() < 0.5, err.max()
