"""moe_dispatch_noalloc against moe_dispatch, through the C ABI.

The no-allocation variant exists for callers that cannot allocate device
memory when they dispatch (a process with a fixed, pre-planned device memory
budget and no workspace to lend, or a latency-critical path that avoids
cudaMalloc because it can synchronise the device).  It keeps its scratch in
a static device array inside the library instead of a caller workspace.

Checked here: two calls in a row (the second one on a different shape, so
any dependence on what the first call left in the shared scratch would
show) give exactly what moe_dispatch gives with a caller workspace -- the
dispatch maps, counts and gathered rows are integer/byte results and must
match bit for bit -- and a request larger than the static scratch is
refused on the host.  This file is collected last so that a run stopping at
its first failure has already run every other test; it also passes alone in
a fresh process.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from block_scaled_fp8_router_gb300 import moe_r3
    return moe_r3


def _case(T, k, E, d, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    ids = torch.argsort(torch.rand((T, E), generator=g, device=DEV), dim=1)[:, :k].to(torch.int32)
    xq = torch.randint(0, 256, (T, d), generator=g, device=DEV, dtype=torch.uint8)
    xs = torch.rand((T, d // 128), generator=g, device=DEV)
    return ids, xq, xs


def _preallocated(T, k, E, d):
    A = T * k
    e = lambda shape, dt: torch.full(shape, -7, dtype=dt, device=DEV) if dt == torch.int32 else \
        torch.zeros(shape, dtype=dt, device=DEV)
    return dict(expert_counts=e((E,), torch.int32), expert_offsets=e((E + 1,), torch.int32),
                sorted_to_slot=e((A,), torch.int32), slot_to_sorted=e((A,), torch.int32),
                rows_sorted=e((A, d), torch.uint8), scales_sorted=e((A, d // 128), torch.float32))


def test_noalloc_matches_workspace_dispatch_twice(L):
    for T, k, E, d, seed in [(3000, 8, 256, 512, 1), (517, 6, 64, 256, 2)]:
        ids, xq, xs = _case(T, k, E, d, seed)
        ref = L.moe_dispatch(ids, E, rows=xq, row_scales=xs)
        out = _preallocated(T, k, E, d)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        L.moe_dispatch_noalloc(ids, E, rows=xq, row_scales=xs, dev_status=st, **out)
        torch.cuda.synchronize()
        assert L.check_status(st) == 0
        n = int(ref[1][-1].item())
        assert n == T * k
        assert torch.equal(out["expert_counts"], ref[0])
        assert torch.equal(out["expert_offsets"], ref[1])
        assert torch.equal(out["sorted_to_slot"][:n], ref[2][:n])
        assert torch.equal(out["slot_to_sorted"], ref[3])
        assert torch.equal(out["rows_sorted"][:n], ref[4][:n])
        assert torch.equal(out["scales_sorted"][:n], ref[5][:n])


def test_noalloc_refuses_oversized_request(L):
    T, k, E = 200000, 8, 1024          # needs far more than the static scratch
    assert L.moe_dispatch_workspace_size(T, k, E) > L.MOE_DISPATCH_NOALLOC_MAX_SCRATCH
    ids = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    with pytest.raises(L.MoEError) as e:
        L.moe_dispatch_noalloc(ids, E)
    assert e.value.status == 4         # MOE_ERR_WORKSPACE, returned before any launch
