"""GPU parity of the one-byte routing payload (pack, unpack, replay from
bytes) against the CPU oracle, through the C ABI: bit-exact bytes, ids and
flags; gates within 1e-5 relative of the oracle and bit-identical to the
int32 replay."""
import numpy as np
import pytest
import torch

from block_scaled_fp8_router_gb300 import synthetic as S
from tests.helpers import bf16_bits

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from block_scaled_fp8_router_gb300 import moe_r3
    return moe_r3


def _ids(n, E, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randint(0, E, (n,), generator=g, device=DEV, dtype=torch.int32)


@pytest.mark.parametrize("n", [0, 1, 15, 16, 17, 1000, 4103, 65536 + 9])
@pytest.mark.parametrize("E", [8, 256])
def test_pack_unpack_bit_exact(L, oracle, n, E):
    ids = _ids(n, E, n + E)
    packed, st = L.moe_payload_pack_u8(ids, E)
    ref, bad = oracle.payload_pack_u8(ids.cpu().numpy(), E)
    assert bad == 0 and L.check_status(st) == 0
    np.testing.assert_array_equal(packed.cpu().numpy(), ref)
    back = L.moe_payload_unpack_u8(packed)
    np.testing.assert_array_equal(back.cpu().numpy(), oracle.payload_unpack_u8(ref))
    assert torch.equal(back, ids)


@pytest.mark.parametrize("off", [1, 3, 8])
def test_pack_unaligned_buffers(L, oracle, off):
    E, n = 200, 3000
    base = _ids(n + 16, E, off)
    ids = base[off:off + n]                              # 4*off bytes past a 16-byte boundary
    out_store = torch.empty(n + 16, dtype=torch.uint8, device=DEV)
    out = out_store[off:off + n]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L._check("pack", L._lib.moe_payload_pack_u8(L._ptr(ids), n, E, L._ptr(out), L._ptr(st), L._stream(None)))
    ref, _ = oracle.payload_pack_u8(ids.cpu().numpy(), E)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)
    back_store = torch.empty(n + 4, dtype=torch.int32, device=DEV)
    back = back_store[1:1 + n]
    L._check("unpack", L._lib.moe_payload_unpack_u8(L._ptr(out), n, L._ptr(back), L._stream(None)))
    assert torch.equal(back, ids)


def test_pack_flags_out_of_range(L, oracle):
    E = 100
    ids = _ids(5000, E, 7)
    ids[[0, 17, 18, 4095, 4999]] = torch.tensor([-1, 100, 255, 256, -2147483648], dtype=torch.int32, device=DEV)
    packed, st = L.moe_payload_pack_u8(ids, E)
    assert L.check_status(st) & L.MOE_DEV_BAD_IDS
    ref, bad = oracle.payload_pack_u8(ids.cpu().numpy(), E)
    assert bad == 5
    np.testing.assert_array_equal(packed.cpu().numpy(), ref)


def test_pack_multilayer_payload_full_size(L, oracle):
    cfg = S.CONFIGS["multilayer_replay"]                  # [8, 8, 16384] ids
    payload = S.make_replay_payload(cfg, DEV)
    packed, st = L.moe_payload_pack_u8(payload, cfg.E)
    ref, bad = oracle.payload_pack_u8(payload.cpu().numpy(), cfg.E)
    assert bad == 0 and L.check_status(st) == 0
    np.testing.assert_array_equal(packed.cpu().numpy(), ref)
    assert torch.equal(L.moe_payload_unpack_u8(packed), payload)


def _route_case(cfg, T):
    x = S.make_x(cfg.with_(T=T), DEV)
    wr = S.make_router_w(cfg, DEV)
    return x, wr


@pytest.mark.parametrize("name,T", [("replay", 2000), ("multilayer_replay", 16384)])
def test_replay_from_bytes_against_oracle(L, oracle, name, T):
    cfg = S.CONFIGS[name].with_(T=T, layers=2)
    payload = S.make_replay_payload(cfg, DEV)
    packed, st = L.moe_payload_pack_u8(payload, cfg.E)
    x, wr = _route_case(cfg, T)
    rl = None
    for l in range(2):
        ids8, g8 = L.moe_route_replay(packed[l], cfg.E, x, wr, cfg.score_fn, 1, 1.0, dev_status=st)
        ids32, g32 = L.moe_route_replay(payload[l], cfg.E, x, wr, cfg.score_fn, 1, 1.0, dev_status=st)
        assert torch.equal(ids8, ids32)
        assert torch.equal(g8.view(torch.int32), g32.view(torch.int32))      # bit for bit
        rid, valid, bad = oracle.replay(oracle.payload_unpack_u8(packed[l].cpu().numpy()), cfg.E)
        assert bad == 0
        np.testing.assert_array_equal(ids8.cpu().numpy(), rid)
        if T <= 2000 or l == 0:
            sample = slice(None) if T <= 2000 else slice(0, T, 61)          # oracle gates on a strided sample
            xs = x[sample]
            rl = oracle.router_logits(bf16_bits(xs), bf16_bits(wr))
            np.testing.assert_allclose(g8[sample].cpu().numpy(),
                                       oracle.gates(rl, rid[sample], cfg.score_fn, 1, 1.0), rtol=1e-5)
    assert L.check_status(st) == 0


def test_replay_from_bytes_flags_bad_ids(L, oracle):
    E, k, T = 200, 4, 300
    cfg = S.CONFIGS["replay"].with_(E=E, k=k, T=T)
    g = torch.Generator(device=DEV).manual_seed(3)
    p = torch.stack([torch.randperm(E, generator=g, device=DEV)[:k] for _ in range(T)], 1).to(torch.uint8)
    p[0, 5] = 230            # id >= E
    p[2, 7] = p[1, 7]        # duplicate within a token
    x, wr = _route_case(cfg, T)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids, gates = L.moe_route_replay(p.contiguous(), E, x, wr, cfg.score_fn, 1, 1.0, dev_status=st)
    assert L.check_status(st) & L.MOE_DEV_BAD_IDS
    rid, valid, bad = oracle.replay(p.cpu().numpy().astype(np.int32), E)
    assert bad == 2
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)
    assert np.all(gates.cpu().numpy()[valid == 0] == 0)
