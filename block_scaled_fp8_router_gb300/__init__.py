"""GB300-native MoE layer with router replay (R3) and block-scaled FP8.

One GPU's Mixture-of-Experts layer as trained in prime-rl ("RL at 1T Scale:
prime-rl Performance Deep Dive", sections "Router replay" and "FP8
training"): router top-k gating or replay of a captured [num_layers, top_k,
seq_len] routing payload, dispatch into expert-contiguous order, a per-expert
SwiGLU FFN as grouped block-scaled FP8 GEMMs, and a gate-weighted combine.

The compute lives in libmoe_r3.so (include/moe_r3.h); ``moe_r3`` is its
binding and ``layer`` composes the calls.  Both are imported on first use,
so ``synthetic`` (input generators) is usable without the library.
"""
from . import synthetic  # noqa: F401

_BINDING = {
    "moe_route_topk", "moe_route_replay", "fp8_block_quant", "moe_dispatch", "moe_dispatch_workspace_size",
    "moe_grouped_ffn_fp8", "moe_grouped_ffn_workspace_size", "moe_combine", "moe_status_str",
    "moe_debug_bounded_wait", "moe_device_sm_count", "check_status", "MoEError",
}
_LAYER = {"MoELayerFP8", "MoEWeightsFP8", "quantize_weights"}


def __getattr__(name):
    if name in _BINDING:
        from . import moe_r3
        return getattr(moe_r3, name)
    if name in _LAYER:
        from . import layer
        return getattr(layer, name)
    raise AttributeError(name)
