"""Pins for the oracle's one-byte routing payload (pack to uint8, unpack).

- exhaustive: every representable id 0..255 with E = 256 maps to its own
  byte and back;
- bounds: every id from -3 to 260 against E in {1, 7, 200, 255, 256},
  enumerated element by element: in range -> its byte, else 0xFF and
  counted;
- structure: a multi-layer [L, k, T] payload keeps its shape and order, and
  replaying an unpacked layer slab equals replaying the original slab.
"""
import numpy as np
import pytest

from block_scaled_fp8_router_gb300 import synthetic as S


def test_pack_every_byte_value(oracle):
    ids = np.arange(256, dtype=np.int32)
    packed, bad = oracle.payload_pack_u8(ids, 256)
    assert bad == 0 and packed.dtype == np.uint8
    assert [int(b) for b in packed] == list(range(256))
    back = oracle.payload_unpack_u8(packed)
    assert back.dtype == np.int32 and [int(v) for v in back] == list(range(256))


@pytest.mark.parametrize("E", [1, 7, 200, 255, 256])
def test_pack_bounds_enumerated(oracle, E):
    ids = np.arange(-3, 261, dtype=np.int32)
    packed, bad = oracle.payload_pack_u8(ids, E)
    n_bad = 0
    for v, b in zip(ids.tolist(), packed.tolist()):
        if 0 <= v < E:
            assert b == v
        else:
            assert b == 0xFF
            n_bad += 1
    assert bad == n_bad == 3 + (261 - E)


def test_pack_multilayer_payload_round_trip(oracle):
    cfg = S.CONFIGS["multilayer_replay"].with_(T=640, layers=3)
    payload = S.make_replay_payload(cfg, "cpu").numpy()      # [L, k, T] int32
    packed, bad = oracle.payload_pack_u8(payload, cfg.E)
    assert bad == 0 and packed.shape == payload.shape and packed.nbytes * 4 == payload.nbytes
    back = oracle.payload_unpack_u8(packed)
    np.testing.assert_array_equal(back, payload)
    for layer in range(cfg.layers):
        a = oracle.replay(payload[layer], cfg.E)
        b = oracle.replay(back[layer], cfg.E)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


def test_pack_empty(oracle):
    packed, bad = oracle.payload_pack_u8(np.zeros((0,), np.int32), 8)
    assert packed.shape == (0,) and bad == 0
    assert oracle.payload_unpack_u8(packed).shape == (0,)
