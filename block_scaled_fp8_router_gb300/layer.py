"""The MoE layer with router replay as one sequence of libmoe_r3 calls.

Sequencing and buffer ownership only: every step is a library kernel.
Buffers are allocated once for a maximum token count and reused, so a
forward pass launches kernels and nothing else (no host sync, no
allocation).  The step order follows the layer of the prime-rl post
("Router replay", "FP8 training"): route or replay -> quantise x (1x128) ->
dispatch -> grouped FP8 SwiGLU FFN -> combine.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import moe_r3 as L


@dataclass
class MoEWeightsFP8:
    w_router: torch.Tensor   # [E, d] bf16
    w13_q: torch.Tensor      # [E, 2F, d] e4m3 codes (rows 0..F-1 gate, F..2F-1 up)
    w13_s: torch.Tensor      # [E, 2F/128, d/128] fp32 scales, or uint8 power-of-two exponents (UE8M0)
    w2_q: torch.Tensor       # [E, d, F] e4m3 codes
    w2_s: torch.Tensor       # [E, d/128, F/128] fp32, or uint8 exponents

    @property
    def ue8m0(self) -> bool:
        """Power-of-two block scales (the block-scaled-MMA variant)."""
        return self.w13_s.dtype == torch.uint8

    @property
    def E(self) -> int:
        return self.w13_q.shape[0]

    def transposed(self):
        """(w2t_q [E, F, d], w2t_s, w13t_q [E, d, 2F], w13t_s): the dgrad GEMMs'
        operands, made once per weight update and cached."""
        if getattr(self, "_t", None) is None:
            w2t = L.fp8_weight_transpose(self.w2_q, self.w2_s)
            w13t = L.fp8_weight_transpose(self.w13_q, self.w13_s)
            self._t = (*w2t, *w13t)
        return self._t

    @property
    def d(self) -> int:
        return self.w13_q.shape[2]

    @property
    def F(self) -> int:
        return self.w13_q.shape[1] // 2


def quantize_weights(w13: torch.Tensor, w2: torch.Tensor, out: MoEWeightsFP8 | None = None, e0: int = 0,
                     ue8m0: bool = False):
    """128x128 block quantisation of bf16 expert weights (once per weight
    update).  w13 [n, 2F, d], w2 [n, d, F] -> codes and scales (fp32, or
    power-of-two exponent bytes with ue8m0 / an `out` holding uint8 scales);
    with `out`, writes experts e0 .. e0+n-1 of it in place."""
    n, twoF, d = w13.shape
    F = twoF // 2
    if out is not None:
        ue8m0 = out.ue8m0
    if ue8m0:
        def quant(src, q=None, s=None):
            return L.fp8_block_quant_ue8m0(src, 128, q=q, scale_exp=s)
    else:
        def quant(src, q=None, s=None):
            return L.fp8_block_quant(src, 128, q=q, scales=s)
    if out is None:
        w13_q, w13_s = quant(w13.reshape(n * twoF, d))
        w2_q, w2_s = quant(w2.reshape(n * d, F))
        return (w13_q.view(n, twoF, d), w13_s.view(n, twoF // 128, d // 128),
                w2_q.view(n, d, F), w2_s.view(n, d // 128, F // 128))
    quant(w13.reshape(n * twoF, d), out.w13_q[e0:e0 + n].view(n * twoF, d),
          out.w13_s[e0:e0 + n].view(n * twoF // 128, d // 128))
    quant(w2.reshape(n * d, F), out.w2_q[e0:e0 + n].view(n * d, F), out.w2_s[e0:e0 + n].view(n * d // 128, F // 128))
    return out


class MoELayerFP8:
    """Forward of one MoE layer on one GPU with preallocated buffers.

    gathered=False: dispatch copies the quantised rows into expert order,
    the grouped FFN reads them there and combine gathers the outputs back.
    gathered=True: dispatch builds the maps only, the FFN gathers its A rows
    from the token-major codes (tile::gather4) and stores its outputs in slot
    order, and combine reads each token's k rows contiguously.  Same bits.
    Weights with power-of-two (UE8M0) scales select the block-scaled-MMA
    variant: x is quantised with power-of-two scales and the FFN is
    moe_grouped_ffn_mx (sorted form).
    """

    def __init__(self, weights: MoEWeightsFP8, T_max: int, k: int, score_fn: int, renorm: int = 1,
                 route_scale: float = 1.0, device=None, gathered: bool = False):
        self.w = weights
        self.gathered = gathered
        self.mx = weights.ue8m0
        if self.mx and gathered:
            raise ValueError("the power-of-two variant runs in the sorted form")
        self.k, self.score_fn, self.renorm, self.route_scale = k, score_fn, renorm, route_scale
        dev = weights.w13_q.device if device is None else device
        E, d, F = weights.E, weights.d, weights.F
        A = T_max * k
        self.T_max = T_max
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
        self.ids = e((T_max, k), torch.int32)
        self.gates = e((T_max, k), torch.float32)
        self.xq = e((T_max, d), torch.uint8)
        self.xs = e((T_max, d // 128), torch.uint8 if self.mx else torch.float32)
        self.counts = e((E,), torch.int32)
        self.offsets = e((E + 1,), torch.int32)
        self.s2s = e((A,), torch.int32)
        self.sl2 = e((A,), torch.int32)
        self.xq_sorted = None if gathered else e((A, d), torch.uint8)
        self.xs_sorted = None if (gathered or self.mx) else e((A, d // 128), torch.float32)
        self.out_sorted = e((A, d), torch.bfloat16)     # slot order when gathered
        self.y = e((T_max, d), torch.bfloat16)
        self.dsp_ws = e((L.moe_dispatch_workspace_size(T_max, k, E),), torch.uint8)
        ws = L.moe_grouped_ffn_mx_workspace_size(A, d, F) if self.mx else L.moe_grouped_ffn_workspace_size(A, d, F)
        self.ffn_ws = e((ws,), torch.uint8)
        self.dev_status = torch.zeros((1,), dtype=torch.int32, device=dev)

    def route(self, x: torch.Tensor, replay_kT: torch.Tensor | None = None, capture_kT: torch.Tensor | None = None):
        T = x.shape[0]
        ids, gates = self.ids[:T], self.gates[:T]
        if replay_kT is None:
            L.moe_route_topk(x, self.w.w_router, self.k, self.score_fn, self.renorm, self.route_scale,
                             topk_ids=ids, topk_gates=gates, capture_kT=capture_kT)
        else:
            L.moe_route_replay(replay_kT, self.w.E, x, self.w.w_router, self.score_fn, self.renorm,
                               self.route_scale, topk_ids=ids, topk_gates=gates, dev_status=self.dev_status)
        return ids, gates

    def forward(self, x: torch.Tensor, replay_kT: torch.Tensor | None = None,
                capture_kT: torch.Tensor | None = None, y: torch.Tensor | None = None,
                train: bool = False) -> torch.Tensor:
        """train=True also keeps GEMM1's pre-activations for backward()."""
        T = x.shape[0]
        if T > self.T_max:
            raise ValueError(f"T={T} exceeds T_max={self.T_max}")
        A = T * self.k
        ids, gates = self.route(x, replay_kT, capture_kT)
        y = self.y[:T] if y is None else y
        if self.mx:
            xq, xe = L.fp8_block_quant_ue8m0(x, 1, q=self.xq[:T], scale_exp=self.xs[:T])
            L.moe_dispatch(ids, self.w.E, rows=xq, expert_counts=self.counts, expert_offsets=self.offsets,
                           sorted_to_slot=self.s2s[:A], slot_to_sorted=self.sl2[:A], rows_sorted=self.xq_sorted[:A],
                           workspace=self.dsp_ws, dev_status=self.dev_status)
            L.moe_grouped_ffn_mx(self.xq_sorted[:A], xe, self.s2s[:A], self.k, self.offsets, self.w.w13_q,
                                 self.w.w13_s, self.w.w2_q, self.w.w2_s, out_sorted=self.out_sorted[:A],
                                 workspace=self.ffn_ws, dev_status=self.dev_status)
            return L.moe_combine(self.out_sorted[:A], self.sl2[:A], gates, y=y)
        xq, xs = L.fp8_block_quant(x, 1, q=self.xq[:T], scales=self.xs[:T])
        if self.gathered:
            L.moe_dispatch(ids, self.w.E, expert_counts=self.counts, expert_offsets=self.offsets,
                           sorted_to_slot=self.s2s[:A], slot_to_sorted=self.sl2[:A], workspace=self.dsp_ws,
                           dev_status=self.dev_status)
            L.moe_grouped_ffn_fp8_gathered(xq, xs, self.k, self.s2s[:A], self.offsets, self.w.w13_q, self.w.w13_s,
                                           self.w.w2_q, self.w.w2_s, out_slots=self.out_sorted[:A],
                                           workspace=self.ffn_ws, dev_status=self.dev_status)
            return L.moe_combine_slots(self.out_sorted[:A], self.sl2[:A], gates, y=y)
        L.moe_dispatch(ids, self.w.E, rows=xq, row_scales=xs, expert_counts=self.counts,
                       expert_offsets=self.offsets, sorted_to_slot=self.s2s[:A], slot_to_sorted=self.sl2[:A],
                       rows_sorted=self.xq_sorted[:A], scales_sorted=self.xs_sorted[:A], workspace=self.dsp_ws,
                       dev_status=self.dev_status)
        if train:
            if getattr(self, "h", None) is None or self.h.shape[0] < A:
                self.h = torch.empty((self.T_max * self.k, 2 * self.w.F), dtype=torch.float32, device=x.device)
            L.moe_grouped_ffn_fp8_train(self.xq_sorted[:A], self.xs_sorted[:A], self.offsets, self.w.w13_q,
                                        self.w.w13_s, self.w.w2_q, self.w.w2_s, self.h[:A],
                                        out_sorted=self.out_sorted[:A], workspace=self.ffn_ws,
                                        dev_status=self.dev_status)
            self._T_train = T
            self._x_train = x
        else:
            L.moe_grouped_ffn_fp8(self.xq_sorted[:A], self.xs_sorted[:A], self.offsets, self.w.w13_q, self.w.w13_s,
                                  self.w.w2_q, self.w.w2_s, out_sorted=self.out_sorted[:A], workspace=self.ffn_ws,
                                  dev_status=self.dev_status)
        return L.moe_combine(self.out_sorted[:A], self.sl2[:A], gates, y=y)

    def backward(self, dy: torch.Tensor, weight_grads: bool = False):
        """Backward of the expert path of the last forward(train=True) with its
        routing fixed (replayed): returns (dx [T, d] bf16 from the experts,
        d_gates [T, k] fp32), and with weight_grads also (dW13 [E, 2F, d],
        dW2 [E, d, F]) fp32.  The router's gradients from these d_gates are
        router_backward's (not part of this call)."""
        T = getattr(self, "_T_train", None)
        if T is None or self.mx or self.gathered:
            raise ValueError("backward needs a forward(train=True) of the fp32-scale sorted form")
        A = T * self.k
        E, d, F = self.w.E, self.w.d, self.w.F
        dev = dy.device
        if getattr(self, "_bw", None) is None:
            e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
            Am = self.T_max * self.k
            self._bw = dict(d_out_q=e((Am, d), torch.uint8), d_out_s=e((Am, d // 128), torch.float32),
                            d_gates=e((self.T_max, self.k), torch.float32), d_act=e((Am, F), torch.bfloat16),
                            dh_q=e((Am, 2 * F), torch.uint8), dh_s=e((Am, 2 * F // 128), torch.float32),
                            dx_sorted=e((Am, d), torch.bfloat16), dx=e((self.T_max, d), torch.bfloat16))
        b = self._bw
        w2t_q, w2t_s, w13t_q, w13t_s = self.w.transposed()
        L.moe_combine_backward(dy, self.gates[:T], self.out_sorted[:A], self.sl2[:A], d_out_q=b["d_out_q"][:A],
                               d_out_s=b["d_out_s"][:A], d_gates=b["d_gates"][:T], dev_status=self.dev_status)
        L.moe_grouped_gemm_fp8(b["d_out_q"][:A], b["d_out_s"][:A], self.offsets, w2t_q, w2t_s, out=b["d_act"][:A],
                               dev_status=self.dev_status)
        L.moe_swiglu_backward(b["d_act"][:A], self.h[:A], dh_q=b["dh_q"][:A], dh_s=b["dh_s"][:A])
        L.moe_grouped_gemm_fp8(b["dh_q"][:A], b["dh_s"][:A], self.offsets, w13t_q, w13t_s, out=b["dx_sorted"][:A],
                               dev_status=self.dev_status)
        dx = L.moe_dispatch_backward(b["dx_sorted"][:A], self.sl2[:A], T, self.k, dx=b["dx"][:T])
        if not weight_grads:
            return dx, b["d_gates"][:T]
        return (dx, b["d_gates"][:T], *self._weight_grads(dy, T))

    def router_backward(self, d_gates: torch.Tensor):
        """Gradients of the router of the last forward(train=True), its ids
        fixed: from d_gates [T, k] (as backward() returns them) ->
        (dx_router [T, d] fp32, the router's part of dL/dx; dW_r [E, d] fp32).
        The full softmax over E (softmax without renormalisation) is not
        supported."""
        T = getattr(self, "_T_train", None)
        if T is None or self.mx or self.gathered:
            raise ValueError("router_backward needs a forward(train=True) of the fp32-scale sorted form")
        A = T * self.k
        if getattr(self, "_rb", None) is None:
            dev = d_gates.device
            self._rb = dict(dl=torch.empty((self.T_max, self.k), dtype=torch.float32, device=dev),
                            dx=torch.empty((self.T_max, self.w.d), dtype=torch.float32, device=dev),
                            dw=torch.empty((self.w.E, self.w.d), dtype=torch.float32, device=dev))
        r = self._rb
        L.moe_router_backward(self._x_train, self.w.w_router, self.ids[:T], d_gates, self.score_fn, self.renorm,
                              self.route_scale, dx=r["dx"][:T], dw_router=r["dw"], sorted_to_slot=self.s2s[:A],
                              expert_offsets=self.offsets, d_logits=r["dl"][:T], dev_status=self.dev_status)
        return r["dx"][:T], r["dw"]

    def _weight_grads(self, dy: torch.Tensor, T: int, events=None):
        """dW13, dW2 of the last train forward; `events` (seven CUDA events, for
        timing) are recorded around the six library calls."""
        rec = (lambda i: events[i].record()) if events else (lambda i: None)
        A = T * self.k
        E, d, F = self.w.E, self.w.d, self.w.F
        dev = dy.device
        ld = L.wgrad_ld(self.T_max * self.k, E)
        if getattr(self, "_wg", None) is None:
            e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
            self._wg = dict(pad=e((E + 1,), torch.int32),
                            aq=e((max(d, 2 * F), ld), torch.uint8), as_=e((max(d, 2 * F) * (ld // 128),), torch.float32),
                            bq=e((max(F, d), ld), torch.uint8), bs=e((max(F, d) * (ld // 128),), torch.float32),
                            dW2=e((E, d, F), torch.float32), dW13=e((E, 2 * F, d), torch.float32))
        w = self._wg
        b = self._bw
        rec(0)
        pad = L.moe_wgrad_pad_offsets(self.offsets, pad=w["pad"])
        s2s = self.s2s[:A]
        # dW2 = d_out^T act
        aq, as_ = L.moe_wgrad_quant(L.WGRAD_SRC_GDY, self.offsets, pad, d, ld, True, dy=dy, gates=self.gates[:T],
                                    sorted_to_slot=s2s, k=self.k, q=w["aq"][:d],
                                    scales=w["as_"][:d * (ld // 128)].view(ld // 128, d))
        rec(1)
        bq, bs = L.moe_wgrad_quant(L.WGRAD_SRC_ACT, self.offsets, pad, F, ld, True, h=self.h, F=F, q=w["bq"][:F],
                                   scales=w["bs"][:F * (ld // 128)].view(ld // 128, F))
        rec(2)
        L.moe_wgrad_gemm(aq, as_, bq, bs, pad, out=w["dW2"], dev_status=self.dev_status)
        rec(3)
        # dW13 = dh^T x
        aq, as_ = L.moe_wgrad_quant(L.WGRAD_SRC_DH, self.offsets, pad, 2 * F, ld, True, h=self.h,
                                    d_act=b["d_act"], F=F, q=w["aq"][:2 * F],
                                    scales=w["as_"][:2 * F * (ld // 128)].view(ld // 128, 2 * F))
        rec(4)
        bq, bs = L.moe_wgrad_quant(L.WGRAD_SRC_X, self.offsets, pad, d, ld, True, x=self._x_train,
                                   sorted_to_slot=s2s, k=self.k, q=w["bq"][:d],
                                   scales=w["bs"][:d * (ld // 128)].view(ld // 128, d))
        rec(5)
        L.moe_wgrad_gemm(aq, as_, bq, bs, pad, out=w["dW13"], dev_status=self.dev_status)
        rec(6)
        return w["dW13"], w["dW2"]


@dataclass
class MoEWeightsNVFP4:
    """NVFP4 expert weights (E2M1 codes two per byte, E4M3 scales per 16
    elements, one fp32 tensor scale per expert matrix) with the scale images
    the NVFP4 GEMM copies to tensor memory."""
    w_router: torch.Tensor   # [E, d] bf16
    w13_q: torch.Tensor      # [E, 2F, d/2]
    w13_s: torch.Tensor      # [E, 2F, d/16] E4M3 block scales
    w13_enc: torch.Tensor    # [E] fp32 tensor scales
    w13_sf: torch.Tensor     # tiled scale images of w13_s
    w2_q: torch.Tensor       # [E, d, F/2]
    w2_s: torch.Tensor       # [E, d, F/16]
    w2_enc: torch.Tensor     # [E]
    w2_sf: torch.Tensor

    @property
    def E(self) -> int:
        return self.w13_q.shape[0]

    @property
    def d(self) -> int:
        return self.w13_q.shape[2] * 2

    @property
    def F(self) -> int:
        return self.w13_q.shape[1] // 2


def quantize_weights_nvfp4(w_router: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor, out=None, e0: int = 0):
    """NVFP4 quantisation of bf16 expert weights w13 [n, 2F, d], w2 [n, d, F],
    one tensor scale per expert matrix (once per weight update).  With `out`
    (an MoEWeightsNVFP4), experts e0 .. e0+n-1 are written in place and the
    scale images are rebuilt by finish_nvfp4_weights."""
    n, twoF, d = w13.shape
    F = twoF // 2
    dev = w13.device
    if out is None:
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
        out = MoEWeightsNVFP4(w_router, e((n, twoF, d // 2), torch.uint8), e((n, twoF, d // 16), torch.uint8),
                              e((n,), torch.float32), None, e((n, d, F // 2), torch.uint8),
                              e((n, d, F // 16), torch.uint8), e((n,), torch.float32), None)
        e0 = 0
    ts = torch.empty((2,), dtype=torch.float32, device=dev)
    for i in range(n):
        L.fp8_quant_nvfp4(w13[i], q=out.w13_q[e0 + i], scales=out.w13_s[e0 + i], tensor_scale=ts)
        out.w13_enc[e0 + i] = ts[0]
        L.fp8_quant_nvfp4(w2[i], q=out.w2_q[e0 + i], scales=out.w2_s[e0 + i], tensor_scale=ts)
        out.w2_enc[e0 + i] = ts[0]
    if out.w13_sf is None or e0 + n == out.E:
        finish_nvfp4_weights(out)
    return out


def finish_nvfp4_weights(w: MoEWeightsNVFP4) -> MoEWeightsNVFP4:
    """(Re)build the tiled scale images of all experts."""
    E, d, F = w.E, w.d, w.F
    w.w13_sf = L.moe_nvfp4_tile_scales(w.w13_s.view(E * 2 * F, d // 16), d, out=w.w13_sf)
    w.w2_sf = L.moe_nvfp4_tile_scales(w.w2_s.view(E * d, F // 16), F, out=w.w2_sf)
    return w


class MoELayerNVFP4:
    """Forward of one MoE layer with NVFP4 activations and expert weights:
    route or replay -> NVFP4 quantisation of x (one tensor scale) -> dispatch
    of the codes and scales -> moe_grouped_ffn_nvfp4 -> combine.  Buffers are
    allocated once for T_max tokens."""

    def __init__(self, weights: MoEWeightsNVFP4, T_max: int, k: int, score_fn: int, renorm: int = 1,
                 route_scale: float = 1.0):
        self.w = weights
        self.k, self.score_fn, self.renorm, self.route_scale = k, score_fn, renorm, route_scale
        dev = weights.w13_q.device
        E, d, F = weights.E, weights.d, weights.F
        if d % 64 != 0:
            raise ValueError("d must be a multiple of 64 (the scales travel as fp32 words)")
        A = T_max * k
        self.T_max = T_max
        e = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
        self.ids = e((T_max, k), torch.int32)
        self.gates = e((T_max, k), torch.float32)
        self.xq = e((T_max, d // 2), torch.uint8)
        self.xs = e((T_max, d // 16), torch.uint8)
        self.x_ts = e((2,), torch.float32)
        self.counts = e((E,), torch.int32)
        self.offsets = e((E + 1,), torch.int32)
        self.s2s = e((A,), torch.int32)
        self.sl2 = e((A,), torch.int32)
        self.xq_sorted = e((A, d // 2), torch.uint8)
        self.xs_sorted = e((A, d // 16), torch.uint8)
        self.out_sorted = e((A, d), torch.bfloat16)
        self.y = e((T_max, d), torch.bfloat16)
        self.dsp_ws = e((L.moe_dispatch_workspace_size(T_max, k, E),), torch.uint8)
        self.ffn_ws = e((L.moe_grouped_ffn_nvfp4_workspace_size(A, d, F),), torch.uint8)
        self.dev_status = torch.zeros((1,), dtype=torch.int32, device=dev)

    def forward(self, x: torch.Tensor, replay_kT: torch.Tensor | None = None, y: torch.Tensor | None = None):
        T = x.shape[0]
        if T > self.T_max:
            raise ValueError(f"T={T} exceeds T_max={self.T_max}")
        A = T * self.k
        d = self.w.d
        ids, gates = self.ids[:T], self.gates[:T]
        if replay_kT is None:
            L.moe_route_topk(x, self.w.w_router, self.k, self.score_fn, self.renorm, self.route_scale,
                             topk_ids=ids, topk_gates=gates)
        else:
            L.moe_route_replay(replay_kT, self.w.E, x, self.w.w_router, self.score_fn, self.renorm,
                               self.route_scale, topk_ids=ids, topk_gates=gates, dev_status=self.dev_status)
        L.fp8_quant_nvfp4(x, q=self.xq[:T], scales=self.xs[:T], tensor_scale=self.x_ts)
        # the E4M3 scale bytes ride with the codes as d/64 fp32 words per row
        L.moe_dispatch(ids, self.w.E, rows=self.xq[:T], row_scales=self.xs[:T].view(torch.float32),
                       expert_counts=self.counts, expert_offsets=self.offsets, sorted_to_slot=self.s2s[:A],
                       slot_to_sorted=self.sl2[:A], rows_sorted=self.xq_sorted[:A],
                       scales_sorted=self.xs_sorted[:A].view(torch.float32), workspace=self.dsp_ws,
                       dev_status=self.dev_status)
        L.moe_grouped_ffn_nvfp4(self.xq_sorted[:A], self.xs_sorted[:A], self.x_ts, self.offsets, self.w.w13_q,
                                self.w.w13_sf, self.w.w13_enc, self.w.w2_q, self.w.w2_sf, self.w.w2_enc,
                                out_sorted=self.out_sorted[:A], workspace=self.ffn_ws, dev_status=self.dev_status)
        y = self.y[:T] if y is None else y
        return L.moe_combine(self.out_sorted[:A], self.sl2[:A], gates, y=y)


class HostStreamer:
    """Forward of a sequence of host batches with the copies overlapped.

    Batch i's x goes host -> device on one copy stream while batch i-1 runs
    on the compute stream, and batch i-1's y goes device -> host on a second
    copy stream while batch i runs; device x / y are double-buffered and
    CUDA events order the three streams.  Host buffers should be pinned.
    Only stream plumbing: every computation is the layer's kernels.
    """

    def __init__(self, layer: MoELayerFP8, T: int):
        self.layer = layer
        dev = layer.y.device
        d = layer.w.d
        self.T = T
        self.xd = [torch.empty((T, d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.yd = [torch.empty((T, d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.h2d = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)
        self.x_ready = [torch.cuda.Event() for _ in range(2)]
        self.y_ready = [torch.cuda.Event() for _ in range(2)]
        self.y_drained = [torch.cuda.Event() for _ in range(2)]

    def run(self, xs_host, ys_host, replays_device=None):
        """xs_host[i] -> forward -> ys_host[i] for every i; returns when all
        copies are enqueued (synchronise the compute / copy streams to wait)."""
        compute = torch.cuda.current_stream()
        n = len(xs_host)
        fresh = [True, True]

        def enqueue_h2d(i):
            b = i & 1
            with torch.cuda.stream(self.h2d):
                if not fresh[b]:
                    self.h2d.wait_event(self.y_ready[b])      # batch i-2 is done reading xd[b]
                self.xd[b].copy_(xs_host[i], non_blocking=True)
                self.x_ready[b].record(self.h2d)

        if n:
            enqueue_h2d(0)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                enqueue_h2d(i + 1)
            compute.wait_event(self.x_ready[b])
            if not fresh[b]:
                compute.wait_event(self.y_drained[b])         # batch i-2's y has left yd[b]
            replay = None if replays_device is None else replays_device[i]
            self.layer.forward(self.xd[b], replay_kT=replay, y=self.yd[b])
            self.y_ready[b].record(compute)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(self.y_ready[b])
                ys_host[i].copy_(self.yd[b], non_blocking=True)
                self.y_drained[b].record(self.d2h)
            fresh[b] = False

    def synchronize(self):
        torch.cuda.current_stream().synchronize()
        self.h2d.synchronize()
        self.d2h.synchronize()
