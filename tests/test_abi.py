"""The C-ABI library loads, exports every entry point include/moe_r3.h
declares, the binding passes every argument at the width the prototype
declares, and the library rejects bad arguments on the host before
launching anything (these calls return before any CUDA API is touched, so
they run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from block_scaled_fp8_router_gb300 import moe_r3
    return moe_r3


def _declared():
    src = open(os.path.join(ROOT, "include", "moe_r3.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+|fp8_\w+)\s*\(", src)))


def test_header_symbols_exported(lib):
    names = _declared()
    assert len(names) >= 10
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(so, n), n
    assert set(names) == set(lib.EXPORTED)


def test_host_side_errors(lib):
    L = lib._lib
    null = None
    # shapes
    assert L.moe_route_topk(null, null, 10, 100, 8, 2, 0, 1, 1.0, null, null, null, null, null) == 2   # d % 128
    assert L.moe_route_topk(null, null, 10, 128, 8, 9, 0, 1, 1.0, null, null, null, null, null) == 2   # k > E
    assert L.moe_route_topk(null, null, 10, 128, 2000, 2, 0, 1, 1.0, null, null, null, null, null) == 2  # E > 1024
    assert L.moe_route_topk(null, null, 10, 128, 8, 2, 5, 1, 1.0, null, null, null, null, null) == 2   # score fn
    assert L.moe_route_topk(null, null, 10, 128, 8, 2, 0, 1, 1.0, null, null, null, null, null) == 1   # NULL
    assert L.moe_route_topk(null, null, 0, 128, 8, 2, 0, 1, 1.0, null, null, null, null, null) == 0    # empty
    x = ctypes.c_void_p(0x1000)
    assert L.moe_route_replay(x, x, x, 10, 128, 8, 2, 0, 0, 1.0, x, x, null, null) == 6   # softmax w/o renorm
    m = ctypes.c_void_p(0x1008)                                                           # 8-byte aligned only
    assert L.moe_route_topk(m, x, 10, 128, 8, 2, 0, 1, 1.0, x, x, null, null, null) == 3
    assert L.moe_route_topk(x, m, 10, 128, 8, 2, 0, 1, 1.0, x, x, null, null, null) == 3
    assert L.moe_route_replay(x, m, x, 10, 128, 8, 2, 1, 1, 1.0, x, x, null, null) == 3
    assert L.moe_route_replay(x, x, m, 10, 128, 8, 2, 1, 1, 1.0, x, x, null, null) == 3
    assert L.moe_route_replay(x, x, null, 10, 128, 8, 2, 1, 1, 1.0, x, x, null, null) == 1  # x without W_r
    # router backward: full softmax unsupported, nulls, dW_r without the maps, alignment, T = 0
    assert L.moe_router_backward(x, x, x, x, 10, 128, 8, 2, 0, 0, 1.0, x, x, null, null, null, null, null) == 6
    assert L.moe_router_backward(x, x, x, null, 10, 128, 8, 2, 1, 1, 1.0, x, x, null, null, null, null, null) == 1
    assert L.moe_router_backward(x, x, x, x, 10, 128, 8, 2, 1, 1, 1.0, x, null, null, x, x, null, null) == 1
    assert L.moe_router_backward(x, x, x, x, 10, 128, 8, 2, 1, 1, 1.0, x, m, null, null, null, null, null) == 3
    assert L.moe_router_backward(x, x, x, x, 10, 100, 8, 2, 1, 1, 1.0, x, x, null, null, null, null, null) == 2
    assert L.moe_router_backward(x, x, x, x, 0, 128, 8, 2, 1, 1, 1.0, x, x, null, null, null, null, null) == 0
    # T = 0 with every [T, .] array NULL (what empty tensors pass) and no dW_r: nothing to do
    assert L.moe_router_backward(null, null, null, null, 0, 128, 8, 2, 1, 1, 1.0, null, null, null, null, null,
                                 null, null) == 0
    assert L.moe_router_backward(null, null, null, null, 0, 128, 8, 2, 1, 1, 1.0, null, null, null, null, m,
                                 null, null) == 3                                       # dW_r misaligned
    assert L.fp8_block_quant(null, 4, 100, 100, 1, null, null, null) == 2
    assert L.fp8_block_quant(null, 4, 128, 128, 128, null, null, null) == 2                 # rows % 128
    assert L.fp8_block_quant(null, 0, 128, 128, 1, null, null, null) == 0
    assert L.fp8_block_quant(ctypes.c_void_p(0x1008), 4, 128, 128, 1, x, x, null) == 3     # misaligned
    ws = L.moe_dispatch_workspace_size(100, 4, 16)
    assert ws > 0
    assert L.moe_dispatch(x, 100, 4, 16, null, 0, null, 0, x, x, x, x, null, null, x, ws - 1, null, null) == 4
    assert L.moe_dispatch(x, 100, 4, 16, null, 0, null, 0, x, x, x, x, null, null, null, ws, null, null) == 4
    assert L.moe_dispatch(x, 100, 4, 16, x, 24, null, 0, x, x, x, x, x, null, x, ws, null, null) == 2  # row_bytes % 16
    assert L.moe_dispatch(x, 100, 33, 64, null, 0, null, 0, x, x, x, x, null, null, x, ws, null, null) == 2
    assert L.moe_combine(null, null, null, 10, 2, 100, null, null) == 2
    assert L.moe_combine(null, null, null, 10, 2, 128, null, null) == 1
    fws = L.moe_grouped_ffn_workspace_size(1000, 256, 512)
    assert fws > 0
    assert L.moe_grouped_ffn_fp8(x, x, x, 1000, 8, 200, 512, x, x, x, x, x, x, fws, null, null) in (2, 6)
    # no rows: nothing launched, every buffer and the workspace may be NULL (what empty tensors pass)
    n7 = [null] * 7
    assert L.moe_grouped_ffn_fp8(null, null, null, 0, 8, 256, 512, *n7[:5], null, 0, null, null) == 0
    assert L.moe_grouped_ffn_fp8_train(null, null, null, 0, 8, 256, 512, *n7[:5], null, null, 0, null, null) == 0
    assert L.moe_grouped_ffn_mx(null, null, null, 0, 8, null, 0, 8, 256, 512, *n7[:5], null, 0, null, null) == 0
    assert L.moe_grouped_ffn_nvfp4(null, null, null, null, 0, 8, 256, 512, *n7[:7], null, 0, null, null) == 0
    assert L.moe_grouped_ffn_fp8_train(x, x, x, 16, 8, 256, 512, x, x, x, x, x, null, x, fws, null, null) == 1
    assert L.moe_grouped_ffn_fp8(x, x, x, 1000, 8, 256, 512, x, x, x, x, x, x, fws - 1, null, null) in (4, 6)
    assert L.moe_payload_pack_u8(x, -1, 8, x, x, null) == 2          # n < 0
    assert L.moe_payload_pack_u8(x, 16, 0, x, x, null) == 2          # E < 1
    assert L.moe_payload_pack_u8(x, 16, 257, x, x, null) == 6        # ids need more than a byte
    assert L.moe_payload_pack_u8(x, 16, 8, x, null, null) == 1       # dev_status required
    assert L.moe_payload_pack_u8(null, 0, 8, null, null, null) == 0  # empty
    assert L.moe_payload_unpack_u8(x, -1, x, null) == 2
    assert L.moe_payload_unpack_u8(null, 16, x, null) == 1
    assert L.moe_route_replay_u8(null, null, null, 10, 100, 8, 2, 1, 1, 1.0, null, null, null, null) == 2
    assert L.moe_route_replay_u8(null, null, null, 10, 128, 8, 2, 1, 1, 1.0, null, null, null, null) == 1
    assert L.moe_debug_bounded_wait(1000, null, null) == 1
    assert L.moe_debug_bounded_wait(-1, x, null) == 2 and L.moe_debug_bounded_wait(10 ** 10 + 1, x, null) == 2
    # backward of the expert path
    y = ctypes.c_void_p(0x1008)                                        # 8-byte aligned only
    assert L.moe_combine_backward(x, x, x, x, 10, 2, 100, 20, x, x, x, null, null) == 2      # d % 128
    assert L.moe_combine_backward(null, null, null, null, 0, 2, 128, 0, null, null, null, null, null) == 0   # empty
    assert L.moe_combine_backward(x, x, x, null, 10, 2, 128, 20, x, x, x, null, null) == 1   # NULL
    assert L.moe_combine_backward(y, x, x, x, 10, 2, 128, 20, x, x, x, null, null) == 3      # misaligned dy
    assert L.moe_swiglu_backward(x, x, 10, 100, x, x, null) == 2                        # F % 128
    assert L.moe_swiglu_backward(null, null, 0, 128, null, null, null) == 0             # empty
    assert L.moe_swiglu_backward(x, x, 10, 128, y, x, null) == 3                        # misaligned dh_q
    assert L.moe_dispatch_backward(x, x, 10, 33, 128, x, null) == 2                     # k > 32
    assert L.moe_dispatch_backward(x, null, 10, 2, 128, x, null) == 1
    assert L.fp8_weight_transpose(x, x, 2, 100, 128, x, x, null) == 2                   # R % 128
    assert L.fp8_weight_transpose(x, x, 0, 128, 128, x, x, null) == 0                   # no experts
    assert L.fp8_weight_transpose(x, x, 2, 128, 128, y, x, null) == 3
    # weight gradients
    assert L.moe_wgrad_pad_offsets(x, 0, x, null) == 2                                  # E < 1
    assert L.moe_wgrad_pad_offsets(null, 4, x, null) == 1
    assert L.moe_wgrad_quant(0, x, x, null, x, 2, null, null, 0, x, x, 4, 100, 256, 1, x, x, null) == 2   # C % 128
    assert L.moe_wgrad_quant(0, x, x, null, x, 2, null, null, 0, x, x, 4, 128, 200, 1, x, x, null) == 2   # ld % 128
    assert L.moe_wgrad_quant(0, x, x, null, x, 40, null, null, 0, x, x, 4, 128, 256, 1, x, x, null) == 2  # k > 32
    assert L.moe_wgrad_quant(5, x, x, x, x, 2, x, x, 128, x, x, 4, 128, 256, 1, x, x, null) == 2          # source
    assert L.moe_wgrad_quant(0, null, x, null, x, 2, null, null, 0, x, x, 4, 128, 256, 1, x, x, null) == 1  # no dy
    assert L.moe_wgrad_quant(1, null, null, null, null, 1, x, null, 128, x, x, 4, 256, 256, 1, x, x, null) == 2  # C != F
    assert L.moe_wgrad_quant(2, null, null, null, null, 1, x, null, 128, x, x, 4, 256, 256, 1, x, x, null) == 1  # no d_act
    assert L.moe_wgrad_quant(2, null, null, null, null, 1, x, x, 128, x, x, 4, 256, 256, 1, y, x, null) == 3    # q
    assert L.moe_wgrad_quant(3, null, null, y, x, 2, null, null, 0, x, x, 4, 128, 256, 1, x, x, null) == 3      # x
    assert L.moe_wgrad_quant(3, null, null, x, x, 2, null, null, 0, x, x, 4, 128, 0, 1, x, x, null) == 0       # ld 0
    assert L.moe_wgrad_gemm(x, x, x, x, x, 4, 200, 256, 256, x, null, null) == 2        # M % 128
    assert L.moe_wgrad_gemm(x, x, x, x, x, 4, 256, 200, 256, x, null, null) == 2        # N % 128
    assert L.moe_wgrad_gemm(x, x, x, x, x, 4, 256, 256, 200, x, null, null) == 2        # ld % 128
    assert L.moe_wgrad_gemm(x, x, x, x, x, 2000, 256, 256, 256, x, null, null) == 2     # E > max
    assert L.moe_wgrad_gemm(x, x, x, x, x, 1024, 1 << 21, 256, 256, x, null, null) == 2  # E * M >= 2^31
    assert L.moe_wgrad_gemm(x, null, x, x, x, 4, 256, 256, 256, x, null, null) == 1
    assert L.moe_wgrad_gemm(x, y, x, x, x, 4, 256, 256, 256, x, null, null) == 3        # a_sT for the bulk copy
    # NVFP4 quantiser
    assert L.fp8_quant_nvfp4(x, 4, 40, x, x, x, null) == 2                              # cols % 16
    assert L.fp8_quant_nvfp4(x, 4, 64, x, x, null, null) == 1                           # tensor scale
    assert L.fp8_quant_nvfp4(null, 4, 64, x, x, x, null) == 1                           # src
    assert L.fp8_quant_nvfp4(y, 4, 64, x, x, x, null) == 3                              # misaligned src
    for s in range(7):
        assert lib.moe_status_str(s)


def _decl_signatures():
    """name -> (return type, [parameter types]) from the header's prototypes."""
    src = open(os.path.join(ROOT, "include", "moe_r3.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for ret, name, params in re.findall(r"^\s*((?:const\s+)?\w+\s*\**)\s*\b((?:moe|fp8)_\w+)\s*\(([^)]*)\)\s*;",
                                        src, flags=re.M):
        types = []
        for prm in params.split(","):
            prm = " ".join(prm.split())
            if prm in ("", "void"):
                continue
            types.append(prm[:prm.rfind("*") + 1] if "*" in prm else prm.rsplit(" ", 1)[0])
        out[name] = (" ".join(ret.split()), types)
    return out


def test_binding_signatures_match_the_header(lib):
    """Every prototype's return and parameter types against the argtypes the
    binding sets (a pointer as a void pointer, int32 as int, int64_t and
    size_t at their own widths), so no argument is passed at the wrong width."""
    want = {"int": ctypes.c_int, "int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t, "float": ctypes.c_float,
            "moe_status": ctypes.c_int}
    sigs = _decl_signatures()
    assert set(sigs) == set(lib.EXPORTED)
    for name, (ret, params) in sigs.items():
        fn = getattr(lib._lib, name)
        assert fn.restype == (ctypes.c_char_p if ret.endswith("*") else want[ret]), name
        assert len(fn.argtypes) == len(params), (name, len(fn.argtypes), len(params))
        for i, (t, a) in enumerate(zip(params, fn.argtypes)):
            assert a == (ctypes.c_void_p if t.endswith("*") else want[t]), (name, i, t, a)
