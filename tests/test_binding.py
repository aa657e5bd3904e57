"""The Python binding rejects tensors of the wrong dtype, shape or device
before it hands anything to the library (these checks run on the host, so
they need no GPU), and the library's status codes become MoEError with the
call's name."""
import pytest
import torch


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from block_scaled_fp8_router_gb300 import moe_r3
    return moe_r3


def test_host_tensors_are_rejected(L):
    x = torch.zeros(8, 128, dtype=torch.bfloat16)              # host memory
    wr = torch.zeros(16, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        L.moe_route_topk(x, wr, 2, 0)
    with pytest.raises(ValueError, match="CUDA"):
        L.fp8_quant_nvfp4(x)
    with pytest.raises(ValueError, match="CUDA"):
        L.moe_payload_pack_u8(torch.zeros(2, 8, dtype=torch.int32), 16)


def test_dtype_and_shape_are_checked(L):
    with pytest.raises(TypeError, match="x: expected torch.bfloat16"):
        L.moe_route_topk(torch.zeros(8, 128, dtype=torch.float32), torch.zeros(16, 128, dtype=torch.bfloat16), 2, 0)
    with pytest.raises(ValueError, match="slot_to_sorted: expected shape"):    # T * k = 16 slots, 15 given
        L.moe_combine(torch.zeros(16, 128, dtype=torch.bfloat16), torch.zeros(15, dtype=torch.int32),
                      torch.zeros(8, 2, dtype=torch.float32))
    with pytest.raises(ValueError, match="contiguous bf16"):
        L.fp8_quant_nvfp4(torch.zeros(8, 128, dtype=torch.float16))
    with pytest.raises(ValueError, match="contiguous int32"):
        L.moe_payload_pack_u8(torch.zeros(2, 8, dtype=torch.int64), 16)
    a_q = torch.zeros(256, 256, dtype=torch.uint8)
    with pytest.raises((TypeError, ValueError)):
        L.moe_wgrad_gemm(a_q, torch.zeros(2, 256), a_q, torch.zeros(2, 256, dtype=torch.float64),
                         torch.zeros(3, dtype=torch.int32))


def test_status_codes_raise_named_errors(L):
    with pytest.raises(L.MoEError) as ei:
        L._check("moe_combine", 2)
    assert "moe_combine" in str(ei.value) and "2" in str(ei.value)
    L._check("moe_combine", 0)                                  # OK passes silently
    for s in range(7):
        assert L.moe_status_str(s)


def test_router_backward_arguments_are_checked(L):
    x = torch.zeros(8, 128, dtype=torch.bfloat16)               # host memory
    wr = torch.zeros(16, 128, dtype=torch.bfloat16)
    ids = torch.zeros(8, 2, dtype=torch.int32)
    dg = torch.zeros(8, 2, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA"):
        L.moe_router_backward(x, wr, ids, dg)
    with pytest.raises(TypeError, match="x: expected torch.bfloat16"):
        L.moe_router_backward(x.float(), wr, ids, dg)
