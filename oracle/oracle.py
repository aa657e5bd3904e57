"""Python face of the CPU oracle (moe_oracle.c): ctypes marshalling only.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers allowed.  The product
library never imports this module, and this module never imports the
product.  All arithmetic lives in ``moe_oracle.c``; here arrays are only
checked for dtype/shape, made contiguous and passed by pointer.

Semantics and citations are in the C file's comments.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_BASE_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so next to it (gcc; OpenMP when the
    compiler has it).  Returns the library path."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    for extra in (["-fopenmp"], []):
        cmd = ["gcc", *_BASE_FLAGS, *extra, "-o", tmp, _SRC, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, _LIB)
            return _LIB
    raise RuntimeError("oracle build failed:\n" + r.stderr)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            F = ctypes.c_float
            sig = {
                "or_bf16_to_f32": (F, [ctypes.c_uint16]),
                "or_f32_to_bf16": (ctypes.c_uint16, [F]),
                "or_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
                "or_e4m3_encode": (ctypes.c_uint8, [F]),
                "or_e2m1_decode": (ctypes.c_double, [ctypes.c_uint8]),
                "or_e2m1_encode": (ctypes.c_uint8, [F]),
                "or_quant_nvfp4": (None, [P, I64, I64, I64, P, P, P]),
                "or_gemm_nvfp4": (None, [P, P, F, P, P, F, I64, I64, I64, P]),
                "or_expert_ffn_nvfp4": (None, [P, P, F, I64, P, I, I, P, P, P, P, P, P, P, P, P, P, P, P]),
                "or_quant_1x128": (None, [P, I64, I64, I64, P, P]),
                "or_quant_128x128": (None, [P, I64, I64, I64, P, P]),
                "or_router_logits": (None, [P, P, I64, I, I, P]),
                "or_topk": (None, [P, I64, I, I, P]),
                "or_gates": (None, [P, P, P, I64, I, I, I, I, F, P]),
                "or_router_backward": (None, [P, P, P, P, P, I64, I, I, I, I, I, F, P, P, P]),
                "or_replay": (I64, [P, I64, I, I, P, P]),
                "or_payload_pack_u8": (I64, [P, I64, I, P]),
                "or_combine_backward": (None, [P, P, P, P, I64, I, I, I64, P, P, P, P]),
                "or_weight_transpose": (None, [P, P, I64, I64, I64, P, P]),
                "or_expert_ffn_preact": (None, [P, P, I64, P, I, I, P, P, P]),
                "or_grouped_gemm": (None, [P, P, I64, P, I64, I64, P, P, P]),
                "or_swiglu_backward": (None, [P, P, I64, I, P, P, P]),
                "or_dispatch_backward": (None, [P, P, I64, I, I, P]),
                "or_pad_offsets": (None, [P, I, P]),
                "or_quant_128x1": (None, [P, P, P, I, I64, P, P]),
                "or_wgrad": (None, [P, P, P, P, P, I, I64, I64, P]),
                "or_payload_unpack_u8": (None, [P, I64, P]),
                "or_dispatch": (I64, [P, I64, I, I, P, P, P, P]),
                "or_gather_rows": (None, [P, I64, P, I64, I, P]),
                "or_fp8_gemm": (None, [P, P, I64, P, P, I64, I64, P]),
                "or_expert_ffn": (None, [P, P, I64, P, I, I, P, P, P, P, P, P, P, P]),
                "or_expert_ffn_rule": (None, [P, P, I64, P, I, I, P, P, P, P, I, P, P, P, P]),
                "or_quant_ue8m0": (None, [P, I64, I64, I64, I, P, P]),
                "or_combine": (None, [P, P, P, I64, I, I, P]),
                "or_num_threads": (I, []),
                "or_set_num_threads": (None, [I]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- scalars

def bf16_to_f32(h: int) -> float:
    return _load().or_bf16_to_f32(h)


def f32_to_bf16(f: float) -> int:
    return _load().or_f32_to_bf16(f)


def e4m3_decode(c: int) -> float:
    return _load().or_e4m3_decode(c)


def e4m3_encode(v: float) -> int:
    return _load().or_e4m3_encode(v)


def num_threads() -> int:
    return _load().or_num_threads()


def set_num_threads(n: int) -> None:
    _load().or_set_num_threads(n)


# ---------------------------------------------------------------- tensors
# bf16 tensors travel as np.uint16 bit patterns, e4m3 as np.uint8 codes.

def quant_1x128(x_bf16: np.ndarray):
    """[rows, cols] bf16 bits -> (codes uint8 [rows, cols], scales f32 [rows, cols/128])."""
    x = _c(x_bf16, np.uint16)
    rows, cols = x.shape
    assert cols % 128 == 0
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 128), np.float32)
    _load().or_quant_1x128(_p(x), rows, cols, cols, _p(q), _p(s))
    return q, s


def quant_128x128(w_bf16: np.ndarray):
    """[rows, cols] bf16 bits -> (codes [rows, cols], scales [rows/128, cols/128])."""
    w = _c(w_bf16, np.uint16)
    rows, cols = w.shape
    assert rows % 128 == 0 and cols % 128 == 0
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows // 128, cols // 128), np.float32)
    _load().or_quant_128x128(_p(w), rows, cols, cols, _p(q), _p(s))
    return q, s


def quant_ue8m0(x_bf16: np.ndarray, block_rows: int):
    """[rows, cols] bf16 bits -> (codes uint8 [rows, cols], biased exponents uint8 [rows/block_rows, cols/128]);
    block scale 2^(e-127), the smallest power of two with amax <= 448 * scale."""
    x = _c(x_bf16, np.uint16)
    rows, cols = x.shape
    assert cols % 128 == 0 and rows % block_rows == 0 and block_rows in (1, 128)
    q = np.empty((rows, cols), np.uint8)
    e = np.empty((rows // block_rows, cols // 128), np.uint8)
    _load().or_quant_ue8m0(_p(x), rows, cols, cols, block_rows, _p(q), _p(e))
    return q, e


def ue8m0_value(e: np.ndarray) -> np.ndarray:
    """Biased exponent bytes -> their scale values 2^(e-127) as fp32 (exact)."""
    return np.ldexp(np.float32(1.0), np.asarray(e, np.int32) - 127).astype(np.float32)


def e2m1_decode(c: int) -> float:
    """FP4 E2M1 code (low 4 bits) -> its value."""
    return _load().or_e2m1_decode(c)


def e2m1_encode(v: float) -> int:
    """binary32 -> E2M1 code, nearest with ties to even, saturating to +-6."""
    return _load().or_e2m1_encode(v)


def quant_nvfp4(x_bf16: np.ndarray):
    """[rows, cols] bf16 bits -> (packed codes uint8 [rows, cols/2], E4M3 block scales uint8 [rows, cols/16],
    s_enc float): 16-element blocks along each row, one fp32 scale for the tensor."""
    x = _c(x_bf16, np.uint16)
    rows, cols = x.shape
    assert cols % 16 == 0
    q = np.empty((rows, cols // 2), np.uint8)
    s = np.empty((rows, cols // 16), np.uint8)
    enc = ctypes.c_float(0.0)
    _load().or_quant_nvfp4(_p(x), rows, cols, cols, _p(q), _p(s), ctypes.byref(enc))
    return q, s, enc.value


def gemm_nvfp4(aq: np.ndarray, as_: np.ndarray, a_enc: float, bq: np.ndarray, bs: np.ndarray, b_enc: float):
    """out [M, N] float64 = a (NVFP4 [M, K]) x b (NVFP4 [N, K])^T from the quant_nvfp4 layouts."""
    aq = _c(aq, np.uint8)
    as_ = _c(as_, np.uint8)
    bq = _c(bq, np.uint8)
    bs = _c(bs, np.uint8)
    M, K = aq.shape[0], aq.shape[1] * 2
    N = bq.shape[0]
    assert bq.shape[1] * 2 == K and as_.shape == (M, K // 16) and bs.shape == (N, K // 16)
    out = np.empty((M, N), np.float64)
    _load().or_gemm_nvfp4(_p(aq), _p(as_), a_enc, _p(bq), _p(bs), b_enc, M, N, K, _p(out))
    return out


def expert_ffn_nvfp4(xq: np.ndarray, xs: np.ndarray, x_enc: float, row_expert: np.ndarray,
                     w13_q: np.ndarray, w13_s: np.ndarray, w13_enc: np.ndarray,
                     w2_q: np.ndarray, w2_s: np.ndarray, w2_enc: np.ndarray):
    """SwiGLU FFN in NVFP4 on sorted rows: x rows (packed [n, d/2], scales [n, d/16], tensor scale x_enc),
    w13 [E, 2F, d/2] / [E, 2F, d/16] / [E], w2 [E, d, F/2] / [E, d, F/16] / [E].
    Returns (h [n, 2F] f32, act bf16 bits [n, F], act_q [n, F/2], act_s [n, F/16], act_enc, out bf16 bits [n, d])."""
    xq = _c(xq, np.uint8)
    xs = _c(xs, np.uint8)
    re = _c(row_expert, np.int32)
    w13_q = _c(w13_q, np.uint8)
    w13_s = _c(w13_s, np.uint8)
    w13_enc = _c(w13_enc, np.float32)
    w2_q = _c(w2_q, np.uint8)
    w2_s = _c(w2_s, np.uint8)
    w2_enc = _c(w2_enc, np.float32)
    n, d = xq.shape[0], xq.shape[1] * 2
    Ew, twoF = w13_q.shape[0], w13_q.shape[1]
    F = twoF // 2
    assert w13_q.shape == (Ew, twoF, d // 2) and w13_s.shape == (Ew, twoF, d // 16) and w13_enc.shape == (Ew,)
    assert w2_q.shape == (Ew, d, F // 2) and w2_s.shape == (Ew, d, F // 16) and w2_enc.shape == (Ew,)
    assert xs.shape == (n, d // 16) and re.shape == (n,) and F % 16 == 0
    if n:
        assert re.min() >= 0 and re.max() < Ew
    h = np.empty((n, twoF), np.float32)
    act = np.empty((n, F), np.uint16)
    act_q = np.empty((n, F // 2), np.uint8)
    act_s = np.empty((n, F // 16), np.uint8)
    act_enc = ctypes.c_float(0.0)
    out = np.empty((n, d), np.uint16)
    _load().or_expert_ffn_nvfp4(_p(xq), _p(xs), x_enc, n, _p(re), d, F, _p(w13_q), _p(w13_s), _p(w13_enc),
                                _p(w2_q), _p(w2_s), _p(w2_enc), _p(h), _p(act), _p(act_q), _p(act_s),
                                ctypes.byref(act_enc), _p(out))
    return h, act, act_q, act_s, act_enc.value, out


def router_logits(x_bf16: np.ndarray, wr_bf16: np.ndarray) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    wr = _c(wr_bf16, np.uint16)
    T, d = x.shape
    E, d2 = wr.shape
    assert d == d2
    out = np.empty((T, E), np.float32)
    _load().or_router_logits(_p(x), _p(wr), T, d, E, _p(out))
    return out


def topk(logits: np.ndarray, k: int) -> np.ndarray:
    l = _c(logits, np.float32)
    T, E = l.shape
    assert 1 <= k <= E
    ids = np.empty((T, k), np.int32)
    _load().or_topk(_p(l), T, E, k, _p(ids))
    return ids


def gates(logits: np.ndarray, ids: np.ndarray, score_fn: int, renorm: int = 1,
          route_scale: float = 1.0, valid: np.ndarray | None = None) -> np.ndarray:
    l = _c(logits, np.float32)
    ids = _c(ids, np.int32)
    T, E = l.shape
    k = ids.shape[1]
    assert k <= 64
    v = None if valid is None else _c(valid, np.uint8)
    g = np.empty((T, k), np.float32)
    _load().or_gates(_p(l), _p(ids), _p(v), T, E, k, score_fn, renorm, route_scale, _p(g))
    return g


def router_backward(x_bf16: np.ndarray, wr_bf16: np.ndarray, ids: np.ndarray, d_gates: np.ndarray,
                    score_fn: int, renorm: int = 1, route_scale: float = 1.0,
                    valid: np.ndarray | None = None, want_dx: bool = True, want_dw: bool = True):
    """Router backward for fixed ids -> (d_logits [T, k], dx [T, d] or None, dw [E, d] or None), fp32."""
    x = _c(x_bf16, np.uint16)
    wr = _c(wr_bf16, np.uint16)
    ids = _c(ids, np.int32)
    dg = _c(d_gates, np.float32)
    T, d = x.shape
    E, d2 = wr.shape
    k = ids.shape[1]
    assert d == d2 and dg.shape == (T, k) and k <= 64
    assert not (score_fn == 0 and not renorm)
    v = None if valid is None else _c(valid, np.uint8)
    dl = np.empty((T, k), np.float32)
    dx = np.empty((T, d), np.float32) if want_dx else None
    dw = np.empty((E, d), np.float32) if want_dw else None
    _load().or_router_backward(_p(x), _p(wr), _p(ids), _p(v), _p(dg), T, d, E, k, score_fn, renorm,
                               route_scale, _p(dl), _p(dx), _p(dw))
    return dl, dx, dw


def replay(payload_kT: np.ndarray, E: int):
    """[k, T] int32 layer slice -> (ids [T, k], valid uint8 [T], n_invalid)."""
    p = _c(payload_kT, np.int32)
    k, T = p.shape
    ids = np.empty((T, k), np.int32)
    valid = np.empty((T,), np.uint8)
    bad = _load().or_replay(_p(p), T, E, k, _p(ids), _p(valid))
    return ids, valid, int(bad)


def payload_pack_u8(ids: np.ndarray, E: int):
    """int32 payload (any shape) -> (uint8 payload of the same shape, number of ids outside [0, E))."""
    a = _c(ids, np.int32)
    out = np.empty(a.shape, np.uint8)
    bad = _load().or_payload_pack_u8(_p(a), a.size, E, _p(out))
    return out, int(bad)


def payload_unpack_u8(p: np.ndarray) -> np.ndarray:
    """uint8 payload (any shape) -> int32 payload of the same shape."""
    a = _c(p, np.uint8)
    out = np.empty(a.shape, np.int32)
    _load().or_payload_unpack_u8(_p(a), a.size, _p(out))
    return out


def combine_backward(dy_bf16: np.ndarray, gates: np.ndarray, out_sorted_bf16: np.ndarray, slot_to_sorted: np.ndarray):
    """Gradients of y = sum_j g * out: (d_out_f [A,d] f32, d_out_q [A,d], d_out_s [A,d/128], d_gates [T,k])."""
    dy = _c(dy_bf16, np.uint16)
    g = _c(gates, np.float32)
    out = _c(out_sorted_bf16, np.uint16)
    sl2 = _c(slot_to_sorted, np.int32)
    T, d = dy.shape
    k = g.shape[1]
    A = out.shape[0]
    d_out_f = np.zeros((A, d), np.float32)
    d_out_q = np.zeros((A, d), np.uint8)
    d_out_s = np.ones((A, d // 128), np.float32)
    d_g = np.empty((T, k), np.float32)
    _load().or_combine_backward(_p(dy), _p(g), _p(out), _p(sl2), T, k, d, A, _p(d_out_f), _p(d_out_q), _p(d_out_s),
                                _p(d_g))
    return d_out_f, d_out_q, d_out_s, d_g


def weight_transpose(q: np.ndarray, s: np.ndarray):
    """[E, R, C] codes + [E, R/128, C/128] scales -> the transposed pair."""
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    E, R, C = q.shape
    qt = np.empty((E, C, R), np.uint8)
    st = np.empty((E, C // 128, R // 128), np.float32)
    _load().or_weight_transpose(_p(q), _p(s), E, R, C, _p(qt), _p(st))
    return qt, st


def expert_ffn_preact(xq: np.ndarray, xs: np.ndarray, row_expert: np.ndarray, w13_q: np.ndarray, w13_s: np.ndarray):
    """GEMM1 pre-activations h = [gate | up] [n, 2F] fp32."""
    xq = _c(xq, np.uint8)
    xs = _c(xs, np.float32)
    re = _c(row_expert, np.int32)
    w13_q = _c(w13_q, np.uint8)
    w13_s = _c(w13_s, np.float32)
    n, d = xq.shape
    F = w13_q.shape[1] // 2
    h = np.empty((n, 2 * F), np.float32)
    _load().or_expert_ffn_preact(_p(xq), _p(xs), n, _p(re), d, F, _p(w13_q), _p(w13_s), _p(h))
    return h


def grouped_gemm(a_q: np.ndarray, a_s: np.ndarray, row_expert: np.ndarray, b_q: np.ndarray, b_s: np.ndarray):
    """out [n, N] bf16 bits = a (rows of expert row_expert[r]) x b[e]^T, b [E, N, K], block-scaled."""
    a_q = _c(a_q, np.uint8)
    a_s = _c(a_s, np.float32)
    re = _c(row_expert, np.int32)
    b_q = _c(b_q, np.uint8)
    b_s = _c(b_s, np.float32)
    n, K = a_q.shape
    N = b_q.shape[1]
    out = np.empty((n, N), np.uint16)
    _load().or_grouped_gemm(_p(a_q), _p(a_s), n, _p(re), K, N, _p(b_q), _p(b_s), _p(out))
    return out


def swiglu_backward(d_act_bf16: np.ndarray, h: np.ndarray):
    """(dh_f [n, 2F] f32, dh_q [n, 2F], dh_s [n, 2F/128]) from the bf16 d_act [n, F] and saved h [n, 2F]."""
    da = _c(d_act_bf16, np.uint16)
    h = _c(h, np.float32)
    n, F = da.shape
    dh_f = np.empty((n, 2 * F), np.float32)
    dh_q = np.empty((n, 2 * F), np.uint8)
    dh_s = np.empty((n, 2 * F // 128), np.float32)
    _load().or_swiglu_backward(_p(da), _p(h), n, F, _p(dh_f), _p(dh_q), _p(dh_s))
    return dh_f, dh_q, dh_s


def dispatch_backward(dx_sorted_bf16: np.ndarray, slot_to_sorted: np.ndarray, T: int, k: int):
    """dx [T, d] bf16 bits = per token the sum of its routed rows' gradients."""
    dxs = _c(dx_sorted_bf16, np.uint16)
    sl2 = _c(slot_to_sorted, np.int32)
    d = dxs.shape[1]
    dx = np.empty((T, d), np.uint16)
    _load().or_dispatch_backward(_p(dxs), _p(sl2), T, k, d, _p(dx))
    return dx


def pad_offsets(offsets: np.ndarray) -> np.ndarray:
    """Expert segments rounded up to 128 rows: pad [E+1] int32."""
    o = _c(offsets, np.int32)
    E = o.shape[0] - 1
    pad = np.empty((E + 1,), np.int32)
    _load().or_pad_offsets(_p(o), E, _p(pad))
    return pad


def quant_128x1(src: np.ndarray, offsets: np.ndarray):
    """fp32 rows [A, C] in expert order -> (codes [C, P] channel-major, scales [C, P/128], pad [E+1])."""
    x = _c(src, np.float32)
    o = _c(offsets, np.int32)
    pad = pad_offsets(o)
    E = o.shape[0] - 1
    C = x.shape[1]
    P = int(pad[E])
    q = np.empty((C, P), np.uint8)
    s = np.ones((C, P // 128), np.float32)
    _load().or_quant_128x1(_p(x), _p(o), _p(pad), E, C, _p(q), _p(s))
    return q, s, pad


def wgrad(a_q: np.ndarray, a_s: np.ndarray, b_q: np.ndarray, b_s: np.ndarray, pad: np.ndarray):
    """Per-expert weight gradient [E, M, N] fp32 from the 128 x 1 layouts a [M, P], b [N, P]."""
    a_q = _c(a_q, np.uint8)
    a_s = _c(a_s, np.float32)
    b_q = _c(b_q, np.uint8)
    b_s = _c(b_s, np.float32)
    pad = _c(pad, np.int32)
    E = pad.shape[0] - 1
    M, N = a_q.shape[0], b_q.shape[0]
    out = np.empty((E, M, N), np.float32)
    _load().or_wgrad(_p(a_q), _p(a_s), _p(b_q), _p(b_s), _p(pad), E, M, N, _p(out))
    return out


def dispatch(ids: np.ndarray, E: int):
    """[T, k] ids -> (counts [E], offsets [E+1], sorted_to_slot [A], slot_to_sorted [A], dropped)."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    A = T * k
    counts = np.empty((E,), np.int32)
    offsets = np.empty((E + 1,), np.int32)
    s2s = np.empty((A,), np.int32)
    sl2 = np.empty((A,), np.int32)
    dropped = _load().or_dispatch(_p(ids), T, k, E, _p(counts), _p(offsets), _p(s2s), _p(sl2))
    return counts, offsets, s2s, sl2, int(dropped)


def gather_rows(rows: np.ndarray, sorted_to_slot: np.ndarray, n_sorted: int, k: int) -> np.ndarray:
    """Rows of any dtype [T, ...] -> rows_sorted [n_sorted, ...]."""
    r = np.ascontiguousarray(rows)
    s2s = _c(sorted_to_slot, np.int32)
    row_bytes = r.strides[0] if r.ndim > 1 else r.itemsize
    out = np.empty((n_sorted,) + r.shape[1:], r.dtype)
    _load().or_gather_rows(_p(r), row_bytes, _p(s2s), n_sorted, k, _p(out))
    return out


def fp8_gemm(a_q: np.ndarray, a_s: np.ndarray, w_q: np.ndarray, w_s: np.ndarray) -> np.ndarray:
    """Block-scaled GEMM: A [M,K] codes + [M,K/128] scales, W [N,K] codes +
    [N/128,K/128] scales -> fp32 [M,N]."""
    a_q = _c(a_q, np.uint8)
    a_s = _c(a_s, np.float32)
    w_q = _c(w_q, np.uint8)
    w_s = _c(w_s, np.float32)
    M, K = a_q.shape
    N = w_q.shape[0]
    assert w_q.shape == (N, K) and a_s.shape == (M, K // 128) and w_s.shape == (N // 128, K // 128)
    out = np.empty((M, N), np.float32)
    _load().or_fp8_gemm(_p(a_q), _p(a_s), M, _p(w_q), _p(w_s), N, K, _p(out))
    return out


def expert_ffn(xq: np.ndarray, xs: np.ndarray, row_expert: np.ndarray,
               w13_q: np.ndarray, w13_s: np.ndarray, w2_q: np.ndarray, w2_s: np.ndarray, ue8m0: bool = False):
    """SwiGLU FFN on sorted rows.  Returns (act_f [n,F] f32, act_q [n,F], act_s [n,F/128], out bf16 [n,d]).
    ue8m0: the act re-quantisation takes power-of-two scales (or_quant_ue8m0's rule)."""
    xq = _c(xq, np.uint8)
    xs = _c(xs, np.float32)
    re = _c(row_expert, np.int32)
    w13_q = _c(w13_q, np.uint8)
    w13_s = _c(w13_s, np.float32)
    w2_q = _c(w2_q, np.uint8)
    w2_s = _c(w2_s, np.float32)
    n, d = xq.shape
    Ew, twoF, d2 = w13_q.shape
    F = twoF // 2
    assert d2 == d and w2_q.shape == (Ew, d, F)
    assert w13_s.shape == (Ew, twoF // 128, d // 128) and w2_s.shape == (Ew, d // 128, F // 128)
    assert xs.shape == (n, d // 128) and re.shape == (n,)
    if n:
        assert re.min() >= 0 and re.max() < Ew
    act_f = np.empty((n, F), np.float32)
    act_q = np.empty((n, F), np.uint8)
    act_s = np.empty((n, F // 128), np.float32)
    out = np.empty((n, d), np.uint16)
    _load().or_expert_ffn_rule(_p(xq), _p(xs), n, _p(re), d, F, _p(w13_q), _p(w13_s), _p(w2_q), _p(w2_s),
                               int(ue8m0),
                          _p(act_f), _p(act_q), _p(act_s), _p(out))
    return act_f, act_q, act_s, out


def combine(out_sorted: np.ndarray, slot_to_sorted: np.ndarray, gates_: np.ndarray) -> np.ndarray:
    o = _c(out_sorted, np.uint16)
    sl2 = _c(slot_to_sorted, np.int32)
    g = _c(gates_, np.float32)
    T, k = g.shape
    d = o.shape[1]
    y = np.empty((T, d), np.uint16)
    _load().or_combine(_p(o), _p(sl2), _p(g), T, k, d, _p(y))
    return y
