"""Python binding of libmoe_r3 (argument marshalling only).

Every function has the name of the C entry point it calls (include/moe_r3.h)
and takes torch CUDA tensors: it checks dtypes and shapes, allocates outputs
the caller did not pass, and hands raw device pointers plus the current CUDA
stream to the library.  All arithmetic runs in the library's kernels; there is
no fallback: if libmoe_r3.so is missing or fails to load, this module raises
on import.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libmoe_r3.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libmoe_r3.so is not built ({_LIB_PATH}); run __graft_entry__.build() first")
_lib = ctypes.CDLL(_LIB_PATH)

P = ctypes.c_void_p
I = ctypes.c_int
I64 = ctypes.c_int64
F = ctypes.c_float
SZ = ctypes.c_size_t

_SIGS = {
    "moe_status_str": (ctypes.c_char_p, [I]),
    "moe_route_topk": (I, [P, P, I, I, I, I, I, I, F, P, P, P, P, P]),
    "moe_route_replay": (I, [P, P, P, I, I, I, I, I, I, F, P, P, P, P]),
    "moe_route_replay_u8": (I, [P, P, P, I, I, I, I, I, I, F, P, P, P, P]),
    "moe_router_backward": (I, [P, P, P, P, I, I, I, I, I, I, F, P, P, P, P, P, P, P]),
    "moe_payload_pack_u8": (I, [P, I64, I, P, P, P]),
    "moe_payload_unpack_u8": (I, [P, I64, P, P]),
    "fp8_block_quant": (I, [P, I64, I64, I64, I, P, P, P]),
    "fp8_block_quant_ue8m0": (I, [P, I64, I64, I64, I, P, P, P]),
    "moe_dispatch_workspace_size": (SZ, [I, I, I]),
    "moe_dispatch": (I, [P, I, I, I, P, I64, P, I, P, P, P, P, P, P, P, SZ, P, P]),
    "moe_dispatch_noalloc": (I, [P, I, I, I, P, I64, P, I, P, P, P, P, P, P, P, P]),
    "moe_grouped_ffn_workspace_size": (SZ, [I64, I, I]),
    "moe_grouped_ffn_fp8": (I, [P, P, P, I64, I, I, I, P, P, P, P, P, P, SZ, P, P]),
    "moe_combine": (I, [P, P, P, I, I, I, P, P]),
    "moe_grouped_ffn_fp8_gathered": (I, [P, P, I, I, P, P, I, I, I, P, P, P, P, P, P, SZ, P, P]),
    "moe_combine_slots": (I, [P, P, P, I, I, I, P, P]),
    "moe_grouped_ffn_mx_workspace_size": (SZ, [I64, I, I]),
    "moe_grouped_ffn_fp8_train": (I, [P, P, P, I64, I, I, I, P, P, P, P, P, P, P, SZ, P, P]),
    "moe_grouped_gemm_fp8": (I, [P, P, P, I64, I, I, I, P, P, P, P, P]),
    "fp8_weight_transpose": (I, [P, P, I64, I64, I64, P, P, P]),
    "moe_combine_backward": (I, [P, P, P, P, I, I, I, I64, P, P, P, P, P]),
    "moe_swiglu_backward": (I, [P, P, I64, I, P, P, P]),
    "moe_dispatch_backward": (I, [P, P, I, I, I, P, P]),
    "moe_wgrad_pad_offsets": (I, [P, I, P, P]),
    "moe_wgrad_quant": (I, [I, P, P, P, P, I, P, P, I, P, P, I, I64, I64, I, P, P, P]),
    "moe_wgrad_gemm": (I, [P, P, P, P, P, I, I, I, I64, P, P, P]),
    "fp8_quant_nvfp4": (I, [P, I64, I64, P, P, P, P]),
    "moe_nvfp4_tiled_scales_size": (SZ, [I64, I64]),
    "moe_nvfp4_tile_scales": (I, [P, I64, I64, P, P]),
    "moe_grouped_ffn_nvfp4_workspace_size": (SZ, [I64, I, I]),
    "moe_grouped_ffn_nvfp4": (I, [P, P, P, P, I64, I, I, I, P, P, P, P, P, P, P, P, SZ, P, P]),
    "moe_grouped_ffn_mx": (I, [P, P, P, I, I, P, I64, I, I, I, P, P, P, P, P, P, SZ, P, P]),
    "moe_debug_bounded_wait": (I, [I64, P, P]),
    "moe_device_sm_count": (I, []),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)
LIB_PATH = _LIB_PATH

MOE_SCORE_SOFTMAX = 0
MOE_SCORE_SIGMOID = 1
MOE_DEV_BAD_IDS = 0x1
MOE_DEV_TIMEOUT = 0x2
MOE_DEV_ROWS = 0x4


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {_lib.moe_status_str(status).decode()} (status {status})")


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MoEError(fn, status)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _want(t: torch.Tensor, dtype, shape, name: str) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _empty(shape, dtype, like: torch.Tensor) -> torch.Tensor:
    return torch.empty(shape, dtype=dtype, device=like.device)


def moe_status_str(status: int) -> str:
    return _lib.moe_status_str(status).decode()


def moe_device_sm_count() -> int:
    return _lib.moe_device_sm_count()


def moe_route_topk(x, w_router, k, score_fn, renorm=1, route_scale=1.0, topk_ids=None, topk_gates=None,
                   capture_kT=None, logits_out=None, stream=None):
    """Router logits (fp32 fma chain) -> top-k ids [T,k] int32, gates [T,k] fp32."""
    T, d = x.shape
    E = w_router.shape[0]
    _want(x, torch.bfloat16, (T, d), "x")
    _want(w_router, torch.bfloat16, (E, d), "w_router")
    topk_ids = _empty((T, k), torch.int32, x) if topk_ids is None else topk_ids
    topk_gates = _empty((T, k), torch.float32, x) if topk_gates is None else topk_gates
    _want(topk_ids, torch.int32, (T, k), "topk_ids")
    _want(topk_gates, torch.float32, (T, k), "topk_gates")
    if capture_kT is not None:
        _want(capture_kT, torch.int32, (k, T), "capture_kT")
    if logits_out is not None:
        _want(logits_out, torch.float32, (T, E), "logits_out")
    _check("moe_route_topk", _lib.moe_route_topk(
        _ptr(x), _ptr(w_router), T, d, E, k, score_fn, renorm, route_scale, _ptr(topk_ids),
        _ptr(topk_gates), _ptr(capture_kT), _ptr(logits_out), _stream(stream)))
    return topk_ids, topk_gates


def moe_route_replay(replay_kT, E, x=None, w_router=None, score_fn=MOE_SCORE_SOFTMAX, renorm=1,
                     route_scale=1.0, topk_ids=None, topk_gates=None, dev_status=None, stream=None):
    """Replay one [k, T] layer slab of the routed-experts payload -> ids [T,k]
    (exact copy) and, when x is given, gates [T,k] from the router logits.
    An int32 slab calls moe_route_replay, a uint8 slab moe_route_replay_u8."""
    k, T = replay_kT.shape
    if replay_kT.dtype == torch.uint8:
        _want(replay_kT, torch.uint8, (k, T), "replay_kT")
        fn_name = "moe_route_replay_u8"
    else:
        _want(replay_kT, torch.int32, (k, T), "replay_kT")
        fn_name = "moe_route_replay"
    topk_ids = _empty((T, k), torch.int32, replay_kT) if topk_ids is None else topk_ids
    _want(topk_ids, torch.int32, (T, k), "topk_ids")
    d = 128
    if x is not None:
        d = x.shape[1]
        _want(x, torch.bfloat16, (T, d), "x")
        _want(w_router, torch.bfloat16, (E, d), "w_router")
        topk_gates = _empty((T, k), torch.float32, x) if topk_gates is None else topk_gates
        _want(topk_gates, torch.float32, (T, k), "topk_gates")
    if dev_status is not None:
        _want(dev_status, torch.int32, (1,), "dev_status")
    _check(fn_name, getattr(_lib, fn_name)(
        _ptr(replay_kT), _ptr(x), _ptr(w_router), T, d, E, k, score_fn, renorm, route_scale, _ptr(topk_ids),
        _ptr(topk_gates), _ptr(dev_status), _stream(stream)))
    return topk_ids, topk_gates


def moe_router_backward(x, w_router, topk_ids, d_gates, score_fn=MOE_SCORE_SIGMOID, renorm=1, route_scale=1.0,
                        dx=True, dw_router=False, sorted_to_slot=None, expert_offsets=None, d_logits=None,
                        dev_status=None, stream=None):
    """Router gradients for fixed ids -> (d_logits [T,k], dx [T,d] or None,
    dw_router [E,d] or None), fp32.  dx / dw_router: True allocates, a tensor
    is written, False / None skips; dw_router needs the dispatch maps."""
    T, d = x.shape
    E = w_router.shape[0]
    k = topk_ids.shape[1]
    _want(x, torch.bfloat16, (T, d), "x")
    _want(w_router, torch.bfloat16, (E, d), "w_router")
    _want(topk_ids, torch.int32, (T, k), "topk_ids")
    _want(d_gates, torch.float32, (T, k), "d_gates")
    d_logits = _empty((T, k), torch.float32, x) if d_logits is None else d_logits
    _want(d_logits, torch.float32, (T, k), "d_logits")
    if dx is True:
        dx = _empty((T, d), torch.float32, x)
    if dx is not None and dx is not False:
        _want(dx, torch.float32, (T, d), "dx")
    else:
        dx = None
    if dw_router is True:
        dw_router = _empty((E, d), torch.float32, x)
    if dw_router is not None and dw_router is not False:
        _want(dw_router, torch.float32, (E, d), "dw_router")
        _want(sorted_to_slot, torch.int32, (T * k,), "sorted_to_slot")
        _want(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    else:
        dw_router = None
    if dev_status is not None:
        _want(dev_status, torch.int32, (1,), "dev_status")
    _check("moe_router_backward", _lib.moe_router_backward(
        _ptr(x), _ptr(w_router), _ptr(topk_ids), _ptr(d_gates), T, d, E, k, score_fn, renorm, route_scale,
        _ptr(d_logits), _ptr(dx), _ptr(sorted_to_slot), _ptr(expert_offsets), _ptr(dw_router), _ptr(dev_status),
        _stream(stream)))
    return d_logits, dx, dw_router


def moe_route_replay_u8(replay_kT, E, **kw):
    """moe_route_replay on a one-byte [k, T] layer slab."""
    if replay_kT.dtype != torch.uint8:
        raise ValueError("replay_kT: uint8 payload slab expected")
    return moe_route_replay(replay_kT, E, **kw)


def moe_payload_pack_u8(ids, E, out=None, dev_status=None, stream=None):
    """int32 routed-experts payload (any shape, contiguous) -> uint8 payload of
    the same shape; out-of-range ids become 0xFF and set MOE_DEV_BAD_IDS in
    dev_status (allocated and zeroed here when not given)."""
    if ids.dtype != torch.int32 or not ids.is_cuda or not ids.is_contiguous():
        raise ValueError("ids: contiguous int32 CUDA tensor")
    out = _empty(tuple(ids.shape), torch.uint8, ids) if out is None else out
    _want(out, torch.uint8, tuple(ids.shape), "out")
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=ids.device)
    _want(dev_status, torch.int32, (1,), "dev_status")
    _check("moe_payload_pack_u8", _lib.moe_payload_pack_u8(
        _ptr(ids), ids.numel(), E, _ptr(out), _ptr(dev_status), _stream(stream)))
    return out, dev_status


def moe_payload_unpack_u8(packed, out=None, stream=None):
    """uint8 payload (any shape, contiguous) -> int32 payload of the same shape."""
    if packed.dtype != torch.uint8 or not packed.is_cuda or not packed.is_contiguous():
        raise ValueError("packed: contiguous uint8 CUDA tensor")
    out = _empty(tuple(packed.shape), torch.int32, packed) if out is None else out
    _want(out, torch.int32, tuple(packed.shape), "out")
    _check("moe_payload_unpack_u8", _lib.moe_payload_unpack_u8(
        _ptr(packed), packed.numel(), _ptr(out), _stream(stream)))
    return out


def fp8_block_quant_ue8m0(src, block_rows, q=None, scale_exp=None, stream=None):
    """bf16 [rows, cols] -> (E4M3 codes uint8 [rows, cols], power-of-two
    scale exponents uint8 [rows/block_rows, cols/128], scale = 2^(e-127))."""
    if src.dim() != 2:
        raise ValueError("src must be 2-D")
    rows, cols = src.shape
    if src.dtype != torch.bfloat16 or not src.is_cuda or src.stride(1) != 1:
        raise ValueError("src: bf16 CUDA tensor with unit column stride")
    q = _empty((rows, cols), torch.uint8, src) if q is None else q
    scale_exp = _empty((rows // block_rows, cols // 128), torch.uint8, src) if scale_exp is None else scale_exp
    _want(q, torch.uint8, (rows, cols), "q")
    _want(scale_exp, torch.uint8, (rows // block_rows, cols // 128), "scale_exp")
    _check("fp8_block_quant_ue8m0", _lib.fp8_block_quant_ue8m0(
        _ptr(src), rows, cols, src.stride(0), block_rows, _ptr(q), _ptr(scale_exp), _stream(stream)))
    return q, scale_exp


def fp8_quant_nvfp4(src, q=None, scales=None, tensor_scale=None, stream=None):
    """bf16 [rows, cols] -> (packed E2M1 codes uint8 [rows, cols/2], E4M3 block
    scales uint8 [rows, cols/16], tensor_scale float32 [2] = (s_enc, amax))."""
    if src.dim() != 2:
        raise ValueError("src must be 2-D")
    rows, cols = src.shape
    if src.dtype != torch.bfloat16 or not src.is_cuda or not src.is_contiguous():
        raise ValueError("src: contiguous bf16 CUDA tensor")
    q = _empty((rows, cols // 2), torch.uint8, src) if q is None else q
    scales = _empty((rows, cols // 16), torch.uint8, src) if scales is None else scales
    tensor_scale = _empty((2,), torch.float32, src) if tensor_scale is None else tensor_scale
    _want(q, torch.uint8, (rows, cols // 2), "q")
    _want(scales, torch.uint8, (rows, cols // 16), "scales")
    _want(tensor_scale, torch.float32, (2,), "tensor_scale")
    _check("fp8_quant_nvfp4", _lib.fp8_quant_nvfp4(_ptr(src), rows, cols, _ptr(q), _ptr(scales), _ptr(tensor_scale),
                                                   _stream(stream)))
    return q, scales, tensor_scale


def fp8_block_quant(src, block_rows, q=None, scales=None, stream=None):
    """bf16 [rows, cols] -> (E4M3 codes uint8 [rows, cols], fp32 scales
    [rows/block_rows, cols/128]); block_rows 1 (activations) or 128 (weights)."""
    if src.dim() != 2:
        raise ValueError("src must be 2-D")
    rows, cols = src.shape
    if src.dtype != torch.bfloat16 or not src.is_cuda or src.stride(1) != 1:
        raise ValueError("src: bf16 CUDA tensor with unit column stride")
    ld = src.stride(0)
    q = _empty((rows, cols), torch.uint8, src) if q is None else q
    scales = _empty((rows // block_rows, cols // 128), torch.float32, src) if scales is None else scales
    _want(q, torch.uint8, (rows, cols), "q")
    _want(scales, torch.float32, (rows // block_rows, cols // 128), "scales")
    _check("fp8_block_quant", _lib.fp8_block_quant(
        _ptr(src), rows, cols, ld, block_rows, _ptr(q), _ptr(scales), _stream(stream)))
    return q, scales


def moe_dispatch_workspace_size(T, k, E) -> int:
    return int(_lib.moe_dispatch_workspace_size(T, k, E))


def moe_dispatch(topk_ids, E, rows=None, row_scales=None, expert_counts=None, expert_offsets=None,
                 sorted_to_slot=None, slot_to_sorted=None, rows_sorted=None, scales_sorted=None,
                 workspace=None, dev_status=None, stream=None):
    """Stable counting sort of the T*k slots by expert and the row gather.
    rows: [T, ...] uint8 (e4m3 codes) or bf16; row_scales: [T, spr] fp32.
    Returns (counts, offsets, sorted_to_slot, slot_to_sorted, rows_sorted, scales_sorted)."""
    T, k = topk_ids.shape
    A = T * k
    _want(topk_ids, torch.int32, (T, k), "topk_ids")
    dev = topk_ids
    expert_counts = _empty((E,), torch.int32, dev) if expert_counts is None else expert_counts
    expert_offsets = _empty((E + 1,), torch.int32, dev) if expert_offsets is None else expert_offsets
    sorted_to_slot = _empty((A,), torch.int32, dev) if sorted_to_slot is None else sorted_to_slot
    slot_to_sorted = _empty((A,), torch.int32, dev) if slot_to_sorted is None else slot_to_sorted
    _want(expert_counts, torch.int32, (E,), "expert_counts")
    _want(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _want(sorted_to_slot, torch.int32, (A,), "sorted_to_slot")
    _want(slot_to_sorted, torch.int32, (A,), "slot_to_sorted")
    row_bytes, spr = 0, 0
    if rows is not None:
        if rows.shape[0] != T or not rows.is_contiguous() or not rows.is_cuda:
            raise ValueError("rows: contiguous CUDA tensor with T rows")
        row_bytes = rows[0].numel() * rows.element_size() if T > 0 else rows.stride(0) * rows.element_size()
        rows_sorted = _empty((A,) + tuple(rows.shape[1:]), rows.dtype, dev) if rows_sorted is None else rows_sorted
        if row_scales is not None:
            spr = row_scales.shape[1]
            _want(row_scales, torch.float32, (T, spr), "row_scales")
            scales_sorted = _empty((A, spr), torch.float32, dev) if scales_sorted is None else scales_sorted
            _want(scales_sorted, torch.float32, (A, spr), "scales_sorted")
    need = moe_dispatch_workspace_size(T, k, E)
    if workspace is None:
        workspace = _empty((need,), torch.uint8, dev)
    _check("moe_dispatch", _lib.moe_dispatch(
        _ptr(topk_ids), T, k, E, _ptr(rows), row_bytes, _ptr(row_scales), spr, _ptr(expert_counts),
        _ptr(expert_offsets), _ptr(sorted_to_slot), _ptr(slot_to_sorted), _ptr(rows_sorted),
        _ptr(scales_sorted), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_status),
        _stream(stream)))
    return expert_counts, expert_offsets, sorted_to_slot, slot_to_sorted, rows_sorted, scales_sorted


MOE_DISPATCH_NOALLOC_MAX_SCRATCH = 4 << 20


def moe_dispatch_noalloc(topk_ids, E, rows=None, row_scales=None, expert_counts=None, expert_offsets=None,
                         sorted_to_slot=None, slot_to_sorted=None, rows_sorted=None, scales_sorted=None,
                         dev_status=None, stream=None):
    """moe_dispatch without a workspace: the library's static device scratch
    is used instead (for callers that cannot allocate device memory at call
    time).  Outputs not passed in are still allocated here by torch; pass
    them all to keep the call allocation-free.  Calls that overlap on the GPU
    share the scratch and race."""
    T, k = topk_ids.shape
    A = T * k
    _want(topk_ids, torch.int32, (T, k), "topk_ids")
    dev = topk_ids
    expert_counts = _empty((E,), torch.int32, dev) if expert_counts is None else expert_counts
    expert_offsets = _empty((E + 1,), torch.int32, dev) if expert_offsets is None else expert_offsets
    sorted_to_slot = _empty((A,), torch.int32, dev) if sorted_to_slot is None else sorted_to_slot
    slot_to_sorted = _empty((A,), torch.int32, dev) if slot_to_sorted is None else slot_to_sorted
    _want(expert_counts, torch.int32, (E,), "expert_counts")
    _want(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _want(sorted_to_slot, torch.int32, (A,), "sorted_to_slot")
    _want(slot_to_sorted, torch.int32, (A,), "slot_to_sorted")
    row_bytes, spr = 0, 0
    if rows is not None:
        if rows.shape[0] != T or not rows.is_contiguous() or not rows.is_cuda:
            raise ValueError("rows: contiguous CUDA tensor with T rows")
        row_bytes = rows[0].numel() * rows.element_size() if T > 0 else rows.stride(0) * rows.element_size()
        rows_sorted = _empty((A,) + tuple(rows.shape[1:]), rows.dtype, dev) if rows_sorted is None else rows_sorted
        if row_scales is not None:
            spr = row_scales.shape[1]
            _want(row_scales, torch.float32, (T, spr), "row_scales")
            scales_sorted = _empty((A, spr), torch.float32, dev) if scales_sorted is None else scales_sorted
            _want(scales_sorted, torch.float32, (A, spr), "scales_sorted")
    _check("moe_dispatch_noalloc", _lib.moe_dispatch_noalloc(
        _ptr(topk_ids), T, k, E, _ptr(rows), row_bytes, _ptr(row_scales), spr, _ptr(expert_counts),
        _ptr(expert_offsets), _ptr(sorted_to_slot), _ptr(slot_to_sorted), _ptr(rows_sorted),
        _ptr(scales_sorted), _ptr(dev_status), _stream(stream)))
    return expert_counts, expert_offsets, sorted_to_slot, slot_to_sorted, rows_sorted, scales_sorted


def moe_grouped_ffn_workspace_size(max_rows, d, F) -> int:
    return int(_lib.moe_grouped_ffn_workspace_size(max_rows, d, F))


def moe_grouped_ffn_fp8(xq_sorted, xs_sorted, expert_offsets, w13_q, w13_s, w2_q, w2_s, out_sorted=None,
                        workspace=None, dev_status=None, stream=None):
    """Per-expert SwiGLU FFN as two grouped block-scaled FP8 GEMMs ->
    out_sorted [max_rows, d] bf16."""
    max_rows, d = xq_sorted.shape
    E, twoF, d2 = w13_q.shape
    F = twoF // 2
    _want(xq_sorted, torch.uint8, (max_rows, d), "xq_sorted")
    _want(xs_sorted, torch.float32, (max_rows, d // 128), "xs_sorted")
    _want(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _want(w13_q, torch.uint8, (E, 2 * F, d), "w13_q")
    _want(w13_s, torch.float32, (E, 2 * F // 128, d // 128), "w13_s")
    _want(w2_q, torch.uint8, (E, d, F), "w2_q")
    _want(w2_s, torch.float32, (E, d // 128, F // 128), "w2_s")
    out_sorted = _empty((max_rows, d), torch.bfloat16, xq_sorted) if out_sorted is None else out_sorted
    _want(out_sorted, torch.bfloat16, (max_rows, d), "out_sorted")
    need = moe_grouped_ffn_workspace_size(max_rows, d, F)
    if workspace is None:
        workspace = _empty((need,), torch.uint8, xq_sorted)
    _check("moe_grouped_ffn_fp8", _lib.moe_grouped_ffn_fp8(
        _ptr(xq_sorted), _ptr(xs_sorted), _ptr(expert_offsets), max_rows, E, d, F, _ptr(w13_q), _ptr(w13_s),
        _ptr(w2_q), _ptr(w2_s), _ptr(out_sorted), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _stream(stream)))
    return out_sorted


def moe_grouped_ffn_fp8_gathered(xq, xs, top_k, sorted_to_slot, expert_offsets, w13_q, w13_s, w2_q, w2_s,
                                 out_slots=None, workspace=None, dev_status=None, stream=None):
    """The grouped FFN reading token-major xq [T, d] / xs [T, d/128] through
    sorted_to_slot and writing out_slots [T*top_k, d] bf16 in slot order."""
    T, d = xq.shape
    k = top_k
    E, twoF, _ = w13_q.shape
    F = twoF // 2
    _want(xq, torch.uint8, (T, d), "xq")
    _want(xs, torch.float32, (T, d // 128), "xs")
    _want(sorted_to_slot, torch.int32, (T * k,), "sorted_to_slot")
    _want(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _want(w13_q, torch.uint8, (E, 2 * F, d), "w13_q")
    _want(w13_s, torch.float32, (E, 2 * F // 128, d // 128), "w13_s")
    _want(w2_q, torch.uint8, (E, d, F), "w2_q")
    _want(w2_s, torch.float32, (E, d // 128, F // 128), "w2_s")
    out_slots = _empty((T * k, d), torch.bfloat16, xq) if out_slots is None else out_slots
    _want(out_slots, torch.bfloat16, (T * k, d), "out_slots")
    if workspace is None:
        workspace = _empty((moe_grouped_ffn_workspace_size(T * k, d, F),), torch.uint8, xq)
    _check("moe_grouped_ffn_fp8_gathered", _lib.moe_grouped_ffn_fp8_gathered(
        _ptr(xq), _ptr(xs), T, k, _ptr(sorted_to_slot), _ptr(expert_offsets), E, d, F, _ptr(w13_q), _ptr(w13_s),
        _ptr(w2_q), _ptr(w2_s), _ptr(out_slots), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _stream(stream)))
    return out_slots


def moe_grouped_ffn_mx_workspace_size(max_rows: int, d: int, F: int) -> int:
    return int(_lib.moe_grouped_ffn_mx_workspace_size(max_rows, d, F))


def moe_grouped_ffn_mx(xq_sorted, x_exp, sorted_to_slot, top_k, expert_offsets, w13_q, w13_exp, w2_q, w2_exp,
                       out_sorted=None, workspace=None, dev_status=None, stream=None):
    """Grouped SwiGLU FFN with power-of-two block scales on the block-scaled
    MMA -> out_sorted [max_rows, d] bf16.  x_exp is token-major [T, d/128]."""
    max_rows, d = xq_sorted.shape
    T = x_exp.shape[0]
    E, twoF, _ = w13_q.shape
    F = twoF // 2
    _want(xq_sorted, torch.uint8, (max_rows, d), "xq_sorted")
    _want(x_exp, torch.uint8, (T, d // 128), "x_exp")
    _want(sorted_to_slot, torch.int32, (sorted_to_slot.numel(),), "sorted_to_slot")
    _want(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _want(w13_q, torch.uint8, (E, 2 * F, d), "w13_q")
    _want(w13_exp, torch.uint8, (E, 2 * F // 128, d // 128), "w13_exp")
    _want(w2_q, torch.uint8, (E, d, F), "w2_q")
    _want(w2_exp, torch.uint8, (E, d // 128, F // 128), "w2_exp")
    out_sorted = _empty((max_rows, d), torch.bfloat16, xq_sorted) if out_sorted is None else out_sorted
    _want(out_sorted, torch.bfloat16, (max_rows, d), "out_sorted")
    if workspace is None:
        workspace = _empty((moe_grouped_ffn_mx_workspace_size(max_rows, d, F),), torch.uint8, xq_sorted)
    _check("moe_grouped_ffn_mx", _lib.moe_grouped_ffn_mx(
        _ptr(xq_sorted), _ptr(x_exp), _ptr(sorted_to_slot), T, top_k, _ptr(expert_offsets), max_rows, E, d, F,
        _ptr(w13_q), _ptr(w13_exp), _ptr(w2_q), _ptr(w2_exp), _ptr(out_sorted), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)))
    return out_sorted


def moe_nvfp4_tiled_scales_size(rows: int, K: int) -> int:
    return int(_lib.moe_nvfp4_tiled_scales_size(rows, K))


def moe_nvfp4_tile_scales(s, K, out=None, stream=None):
    """E4M3 block scales [rows, K/16] of an NVFP4 weight matrix -> the scale
    images the NVFP4 GEMM copies to tensor memory (uint8, flat)."""
    rows = s.shape[0]
    _want(s, torch.uint8, (rows, K // 16), "s")
    n = moe_nvfp4_tiled_scales_size(rows, K)
    out = _empty((n,), torch.uint8, s) if out is None else out
    _want(out, torch.uint8, (n,), "out")
    _check("moe_nvfp4_tile_scales", _lib.moe_nvfp4_tile_scales(_ptr(s), rows, K, _ptr(out), _stream(stream)))
    return out


def moe_grouped_ffn_nvfp4_workspace_size(max_rows: int, d: int, F: int) -> int:
    return int(_lib.moe_grouped_ffn_nvfp4_workspace_size(max_rows, d, F))


def moe_grouped_ffn_nvfp4(xq_sorted, xs_sorted, x_enc, expert_offsets, w13_q, w13_sf_tiled, w13_enc, w2_q,
                          w2_sf_tiled, w2_enc, out_sorted=None, workspace=None, dev_status=None, stream=None):
    """Grouped SwiGLU FFN in NVFP4 -> out_sorted [max_rows, d] bf16.  xq_sorted
    [max_rows, d/2] E2M1 codes, xs_sorted [max_rows, d/16] E4M3 scales, x_enc
    (one device float: the token tensor's s_enc); w13_q [E, 2F, d/2], w2_q
    [E, d, F/2] with their tiled scale images and per-expert s_enc [E]."""
    max_rows, dh = xq_sorted.shape
    d = 2 * dh
    E, twoF, _ = w13_q.shape
    F = twoF // 2
    _want(xq_sorted, torch.uint8, (max_rows, d // 2), "xq_sorted")
    _want(xs_sorted, torch.uint8, (max_rows, d // 16), "xs_sorted")
    if x_enc.dtype != torch.float32 or x_enc.numel() < 1 or not x_enc.is_cuda:
        raise ValueError("x_enc: float32 CUDA tensor (its first element is the tensor scale)")
    _want(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _want(w13_q, torch.uint8, (E, 2 * F, d // 2), "w13_q")
    _want(w13_sf_tiled, torch.uint8, (moe_nvfp4_tiled_scales_size(E * 2 * F, d),), "w13_sf_tiled")
    _want(w13_enc, torch.float32, (E,), "w13_enc")
    _want(w2_q, torch.uint8, (E, d, F // 2), "w2_q")
    _want(w2_sf_tiled, torch.uint8, (moe_nvfp4_tiled_scales_size(E * d, F),), "w2_sf_tiled")
    _want(w2_enc, torch.float32, (E,), "w2_enc")
    out_sorted = _empty((max_rows, d), torch.bfloat16, xq_sorted) if out_sorted is None else out_sorted
    _want(out_sorted, torch.bfloat16, (max_rows, d), "out_sorted")
    if workspace is None:
        workspace = _empty((moe_grouped_ffn_nvfp4_workspace_size(max_rows, d, F),), torch.uint8, xq_sorted)
    _check("moe_grouped_ffn_nvfp4", _lib.moe_grouped_ffn_nvfp4(
        _ptr(xq_sorted), _ptr(xs_sorted), _ptr(x_enc), _ptr(expert_offsets), max_rows, E, d, F, _ptr(w13_q),
        _ptr(w13_sf_tiled), _ptr(w13_enc), _ptr(w2_q), _ptr(w2_sf_tiled), _ptr(w2_enc), _ptr(out_sorted),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)))
    return out_sorted


def moe_grouped_ffn_fp8_train(xq_sorted, xs_sorted, expert_offsets, w13_q, w13_s, w2_q, w2_s, h_out,
                              out_sorted=None, workspace=None, dev_status=None, stream=None):
    """moe_grouped_ffn_fp8 that also writes GEMM1's pre-activations h [max_rows, 2F] fp32."""
    max_rows, d = xq_sorted.shape
    E, twoF, _ = w13_q.shape
    F = twoF // 2
    _want(xq_sorted, torch.uint8, (max_rows, d), "xq_sorted")
    _want(xs_sorted, torch.float32, (max_rows, d // 128), "xs_sorted")
    _want(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _want(h_out, torch.float32, (max_rows, 2 * F), "h_out")
    out_sorted = _empty((max_rows, d), torch.bfloat16, xq_sorted) if out_sorted is None else out_sorted
    _want(out_sorted, torch.bfloat16, (max_rows, d), "out_sorted")
    if workspace is None:
        workspace = _empty((moe_grouped_ffn_workspace_size(max_rows, d, F),), torch.uint8, xq_sorted)
    _check("moe_grouped_ffn_fp8_train", _lib.moe_grouped_ffn_fp8_train(
        _ptr(xq_sorted), _ptr(xs_sorted), _ptr(expert_offsets), max_rows, E, d, F, _ptr(w13_q), _ptr(w13_s),
        _ptr(w2_q), _ptr(w2_s), _ptr(out_sorted), _ptr(h_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)))
    return out_sorted


def moe_grouped_gemm_fp8(a_q, a_s, expert_offsets, b_q, b_s, out=None, dev_status=None, stream=None):
    """Grouped block-scaled FP8 GEMM, bf16 out [max_rows, N] = a [max_rows, K] x b[e]^T, b [E, N, K]."""
    max_rows, K = a_q.shape
    E, N, _ = b_q.shape
    _want(a_q, torch.uint8, (max_rows, K), "a_q")
    _want(a_s, torch.float32, (max_rows, K // 128), "a_s")
    _want(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _want(b_q, torch.uint8, (E, N, K), "b_q")
    _want(b_s, torch.float32, (E, N // 128, K // 128), "b_s")
    out = _empty((max_rows, N), torch.bfloat16, a_q) if out is None else out
    _want(out, torch.bfloat16, (max_rows, N), "out")
    _check("moe_grouped_gemm_fp8", _lib.moe_grouped_gemm_fp8(
        _ptr(a_q), _ptr(a_s), _ptr(expert_offsets), max_rows, E, K, N, _ptr(b_q), _ptr(b_s), _ptr(out),
        _ptr(dev_status), _stream(stream)))
    return out


def fp8_weight_transpose(q, s, qt=None, st=None, stream=None):
    """[E, R, C] codes + [E, R/128, C/128] scales -> transposed [E, C, R] / [E, C/128, R/128]."""
    E, R, C = q.shape
    _want(q, torch.uint8, (E, R, C), "q")
    _want(s, torch.float32, (E, R // 128, C // 128), "s")
    qt = _empty((E, C, R), torch.uint8, q) if qt is None else qt
    st = _empty((E, C // 128, R // 128), torch.float32, q) if st is None else st
    _want(qt, torch.uint8, (E, C, R), "qt")
    _want(st, torch.float32, (E, C // 128, R // 128), "st")
    _check("fp8_weight_transpose", _lib.fp8_weight_transpose(_ptr(q), _ptr(s), E, R, C, _ptr(qt), _ptr(st),
                                                             _stream(stream)))
    return qt, st


def moe_combine_backward(dy, gates, out_sorted, slot_to_sorted, d_out_q=None, d_out_s=None, d_gates=None,
                         dev_status=None, stream=None):
    """-> (d_out_q [A, d] e4m3, d_out_s [A, d/128], d_gates [T, k])."""
    T, k = gates.shape
    A, d = out_sorted.shape
    _want(dy, torch.bfloat16, (T, d), "dy")
    _want(gates, torch.float32, (T, k), "gates")
    _want(out_sorted, torch.bfloat16, (A, d), "out_sorted")
    _want(slot_to_sorted, torch.int32, (T * k,), "slot_to_sorted")
    d_out_q = _empty((A, d), torch.uint8, dy) if d_out_q is None else d_out_q
    d_out_s = _empty((A, d // 128), torch.float32, dy) if d_out_s is None else d_out_s
    d_gates = _empty((T, k), torch.float32, dy) if d_gates is None else d_gates
    _want(d_out_q, torch.uint8, (A, d), "d_out_q")
    _want(d_out_s, torch.float32, (A, d // 128), "d_out_s")
    _want(d_gates, torch.float32, (T, k), "d_gates")
    _check("moe_combine_backward", _lib.moe_combine_backward(
        _ptr(dy), _ptr(gates), _ptr(out_sorted), _ptr(slot_to_sorted), T, k, d, A, _ptr(d_out_q), _ptr(d_out_s),
        _ptr(d_gates), _ptr(dev_status), _stream(stream)))
    return d_out_q, d_out_s, d_gates


def moe_swiglu_backward(d_act, h, dh_q=None, dh_s=None, stream=None):
    """bf16 d_act [rows, F], fp32 h [rows, 2F] -> (dh_q [rows, 2F] e4m3, dh_s [rows, 2F/128])."""
    rows, F = d_act.shape
    _want(d_act, torch.bfloat16, (rows, F), "d_act")
    _want(h, torch.float32, (rows, 2 * F), "h")
    dh_q = _empty((rows, 2 * F), torch.uint8, d_act) if dh_q is None else dh_q
    dh_s = _empty((rows, 2 * F // 128), torch.float32, d_act) if dh_s is None else dh_s
    _want(dh_q, torch.uint8, (rows, 2 * F), "dh_q")
    _want(dh_s, torch.float32, (rows, 2 * F // 128), "dh_s")
    _check("moe_swiglu_backward", _lib.moe_swiglu_backward(_ptr(d_act), _ptr(h), rows, F, _ptr(dh_q), _ptr(dh_s),
                                                           _stream(stream)))
    return dh_q, dh_s


def moe_dispatch_backward(dx_sorted, slot_to_sorted, T, k, dx=None, stream=None):
    """dx [T, d] bf16 = per token the sum of its routed rows' gradients."""
    A, d = dx_sorted.shape
    if dx_sorted.dtype != torch.bfloat16 or not dx_sorted.is_contiguous():
        raise ValueError("dx_sorted: contiguous bf16")
    _want(slot_to_sorted, torch.int32, (T * k,), "slot_to_sorted")
    dx = _empty((T, d), torch.bfloat16, dx_sorted) if dx is None else dx
    _want(dx, torch.bfloat16, (T, d), "dx")
    _check("moe_dispatch_backward", _lib.moe_dispatch_backward(_ptr(dx_sorted), _ptr(slot_to_sorted), T, k, d,
                                                               _ptr(dx), _stream(stream)))
    return dx


WGRAD_SRC_GDY, WGRAD_SRC_ACT, WGRAD_SRC_DH, WGRAD_SRC_X = 0, 1, 2, 3


def wgrad_ld(max_rows: int, E: int) -> int:
    """A host-side bound of the padded row extent (multiple of 128)."""
    return ((max_rows + 127) // 128 + E) * 128


def moe_wgrad_pad_offsets(expert_offsets, pad=None, stream=None):
    E = expert_offsets.numel() - 1
    pad = _empty((E + 1,), torch.int32, expert_offsets) if pad is None else pad
    _want(pad, torch.int32, (E + 1,), "pad")
    _check("moe_wgrad_pad_offsets", _lib.moe_wgrad_pad_offsets(_ptr(expert_offsets), E, _ptr(pad), _stream(stream)))
    return pad


def moe_wgrad_quant(src, expert_offsets, pad, C, ld, kb_major, dy=None, gates=None, x=None, sorted_to_slot=None,
                    k=1, h=None, d_act=None, F=0, q=None, scales=None, stream=None):
    """One weight-gradient operand, 128 x 1 quantised, channel-major: (q [C, ld], scales)."""
    E = expert_offsets.numel() - 1
    dev = expert_offsets.device
    q = torch.empty((C, ld), dtype=torch.uint8, device=dev) if q is None else q
    sshape = (ld // 128, C) if kb_major else (C, ld // 128)
    scales = torch.empty(sshape, dtype=torch.float32, device=dev) if scales is None else scales
    _want(q, torch.uint8, (C, ld), "q")
    _want(scales, torch.float32, sshape, "scales")
    _check("moe_wgrad_quant", _lib.moe_wgrad_quant(
        src, _ptr(dy), _ptr(gates), _ptr(x), _ptr(sorted_to_slot), k, _ptr(h), _ptr(d_act), F,
        _ptr(expert_offsets), _ptr(pad), E, C, ld, int(kb_major), _ptr(q), _ptr(scales), _stream(stream)))
    return q, scales


def moe_wgrad_gemm(a_q, a_sT, b_q, b_sT, pad, out=None, dev_status=None, stream=None):
    """out [E, M, N] fp32: per expert the weight gradient over its rows
    (both operands' scales kb-major, [ld/128, M] and [ld/128, N])."""
    M, ld = a_q.shape
    N = b_q.shape[0]
    E = pad.numel() - 1
    _want(a_q, torch.uint8, (M, ld), "a_q")
    _want(a_sT, torch.float32, (ld // 128, M), "a_sT")
    _want(b_q, torch.uint8, (N, ld), "b_q")
    _want(b_sT, torch.float32, (ld // 128, N), "b_sT")
    out = _empty((E, M, N), torch.float32, a_q) if out is None else out
    _want(out, torch.float32, (E, M, N), "out")
    _check("moe_wgrad_gemm", _lib.moe_wgrad_gemm(_ptr(a_q), _ptr(a_sT), _ptr(b_q), _ptr(b_sT), _ptr(pad), E, M, N, ld,
                                                 _ptr(out), _ptr(dev_status), _stream(stream)))
    return out


def moe_combine_slots(out_slots, slot_to_sorted, gates, y=None, stream=None):
    """moe_combine over expert rows stored in slot order [T*k, d]."""
    T, k = gates.shape
    d = out_slots.shape[1]
    _want(out_slots, torch.bfloat16, (T * k, d), "out_slots")
    _want(slot_to_sorted, torch.int32, (T * k,), "slot_to_sorted")
    _want(gates, torch.float32, (T, k), "gates")
    y = _empty((T, d), torch.bfloat16, out_slots) if y is None else y
    _want(y, torch.bfloat16, (T, d), "y")
    _check("moe_combine_slots", _lib.moe_combine_slots(
        _ptr(out_slots), _ptr(slot_to_sorted), _ptr(gates), T, k, d, _ptr(y), _stream(stream)))
    return y


def moe_combine(out_sorted, slot_to_sorted, gates, y=None, stream=None):
    """y [T, d] bf16 = gate-weighted sum of each token's k expert rows."""
    T, k = gates.shape
    d = out_sorted.shape[1]
    if out_sorted.dtype != torch.bfloat16 or not out_sorted.is_contiguous():
        raise ValueError("out_sorted: contiguous bf16")
    _want(slot_to_sorted, torch.int32, (T * k,), "slot_to_sorted")
    _want(gates, torch.float32, (T, k), "gates")
    y = _empty((T, d), torch.bfloat16, out_sorted) if y is None else y
    _want(y, torch.bfloat16, (T, d), "y")
    _check("moe_combine", _lib.moe_combine(
        _ptr(out_sorted), _ptr(slot_to_sorted), _ptr(gates), T, k, d, _ptr(y), _stream(stream)))
    return y


def moe_debug_bounded_wait(timeout_ns, dev_status, stream=None):
    _want(dev_status, torch.int32, (1,), "dev_status")
    _check("moe_debug_bounded_wait", _lib.moe_debug_bounded_wait(timeout_ns, _ptr(dev_status), _stream(stream)))


def check_status(dev_status: torch.Tensor) -> int:
    """Read the device status word (synchronises with the current stream)."""
    return int(dev_status.item())
