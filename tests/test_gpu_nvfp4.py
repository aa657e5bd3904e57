"""GPU parity of the NVFP4 quantiser (fp8_quant_nvfp4) against the CPU
oracle, bit for bit: the packed E2M1 codes, the E4M3 block scales and the
tensor scale, on inputs with block magnitudes across the E4M3 scale range
(normal and subnormal block scales), all-zero blocks, signed zeros,
elements on E2M1 rounding midpoints, an all-zero tensor and an empty one."""
import numpy as np
import pytest
import torch

from tests.helpers import bf16_bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from block_scaled_fp8_router_gb300 import moe_r3
    return moe_r3


@pytest.fixture(scope="module")
def oracle():
    from oracle import oracle as O
    return O


def _input(rows, cols, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g) * torch.exp2(
        torch.randint(-12, 7, (rows, cols // 16), generator=g).float()).repeat_interleave(16, dim=1)
    x[0, :16] = 0.0                                   # an all-zero block
    x[0, 16:32] = -0.0                                # signed zeros
    # a block whose scaled values sit on E2M1 midpoints: max 6 * 2^-3 = 0.75
    x[1, :16] = torch.tensor([0.75, 0.03125, 0.09375, 0.15625, 0.21875, 0.3125, 0.4375, 0.625,
                              -0.75, -0.03125, -0.09375, -0.15625, -0.21875, -0.3125, -0.4375, -0.625])
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("rows,cols,seed", [(1, 16, 1), (37, 272, 2), (256, 2048, 3), (1000, 7168, 4)])
def test_nvfp4_quant_bit_exact(L, oracle, rows, cols, seed):
    xb = _input(rows, cols, seed) if rows > 1 else torch.randn(rows, cols).to(torch.bfloat16)
    q, s, ts = L.fp8_quant_nvfp4(xb.to(DEV))
    torch.cuda.synchronize()
    oq, os_, oenc = oracle.quant_nvfp4(bf16_bits(xb))
    assert ts[0].item() == oenc
    assert ts[1].item() == xb.float().abs().max().item()
    np.testing.assert_array_equal(s.cpu().numpy(), os_)
    np.testing.assert_array_equal(q.cpu().numpy(), oq)


def test_nvfp4_quant_zero_and_empty(L, oracle):
    z = torch.zeros(4, 64, dtype=torch.bfloat16, device=DEV)
    q, s, ts = L.fp8_quant_nvfp4(z)
    torch.cuda.synchronize()
    assert ts[0].item() == 1.0 and ts[1].item() == 0.0
    assert torch.all(q == 0) and torch.all(s == 0)
    e = torch.zeros(0, 64, dtype=torch.bfloat16, device=DEV)
    q, s, ts = L.fp8_quant_nvfp4(e)
    torch.cuda.synchronize()
    assert q.shape == (0, 32) and s.shape == (0, 4) and ts[0].item() == 1.0


def test_nvfp4_quant_rounding_midpoints(L, oracle):
    """A tensor whose scales are exact (amax 0.75: s_enc = 3584, block scale
    448, element scale 8), so the scaled values 0.25, 0.75, ..., 5 sit on
    E2M1 rounding midpoints and the ties-to-even rule decides every code."""
    x = torch.zeros(2, 32)
    mid = torch.tensor([0.75, 0.03125, 0.09375, 0.15625, 0.21875, 0.3125, 0.4375, 0.625])
    x[1, :16] = torch.cat([mid, -mid])
    x[1, 16:32] = torch.cat([-mid, mid])
    xb = x.to(torch.bfloat16)
    q, s, ts = L.fp8_quant_nvfp4(xb.to(DEV))
    torch.cuda.synchronize()
    oq, os_, oenc = oracle.quant_nvfp4(bf16_bits(xb))
    assert oenc == 3584.0 and ts[0].item() == oenc
    np.testing.assert_array_equal(s.cpu().numpy(), os_)
    np.testing.assert_array_equal(q.cpu().numpy(), oq)
