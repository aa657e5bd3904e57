"""HostStreamer (host batches in, host results out, copies overlapped with
compute) gives exactly what the plain layer forward gives."""
import pytest
import torch

from block_scaled_fp8_router_gb300 import synthetic as S

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def test_streamer_matches_forward():
    import __graft_entry__
    __graft_entry__.build()
    from block_scaled_fp8_router_gb300.layer import HostStreamer, MoELayerFP8, MoEWeightsFP8, quantize_weights
    cfg = S.CONFIGS["tiny"]
    layer = MoELayerFP8(MoEWeightsFP8(S.make_router_w(cfg, DEV), *quantize_weights(S.make_w13(cfg, DEV),
                                                                                   S.make_w2(cfg, DEV))),
                        cfg.T, cfg.k, cfg.score_fn)
    xs = [S.make_x(cfg, "cpu", seed=s).pin_memory() for s in range(5)]
    ys = [torch.empty_like(x).pin_memory() for x in xs]
    st = HostStreamer(layer, cfg.T)
    st.run(xs, ys)
    st.synchronize()
    for x, y in zip(xs, ys):
        ref = layer.forward(x.to(DEV)).cpu()
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
