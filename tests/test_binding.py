"""The Python binding's argument checks.

The binding hands raw pointers to the C library, whose contract is device
memory on the current device.  Tensors it cannot take (host tensors, the
wrong dtype or shape, tensors on different devices) must raise ValueError in
Python before any pointer reaches a kernel.  The CPU tests run without a GPU
and without loading the library; the GPU tests mix one host tensor into
otherwise valid CUDA arguments.
"""
import pytest

import tensor_core_tiled_02_gb300 as tc

torch = pytest.importorskip("torch")


def test_host_operands_rejected():
    a = torch.zeros((128, 64), dtype=torch.float16)
    b = torch.zeros((64, 128), dtype=torch.float16)
    with pytest.raises(ValueError):
        tc.matmul(a, b)
    with pytest.raises(ValueError):
        tc.matmul_acc(a, b, torch.zeros((128, 128), dtype=torch.float16))
    with pytest.raises(ValueError):
        tc.add_matrices(torch.zeros((32, 256)), torch.zeros((32, 256)))


@pytest.mark.parametrize("bad", ["dtype", "inner", "rank", "out_dtype"])
def test_malformed_operands_rejected(bad):
    a = torch.zeros((128, 64), dtype=torch.float16)
    b = torch.zeros((64, 128), dtype=torch.float16)
    kw = {}
    if bad == "dtype":
        a = a.float()
    elif bad == "inner":
        b = torch.zeros((72, 128), dtype=torch.float16)
    elif bad == "rank":
        a = a.reshape(2, 64, 64)
    else:
        kw["out_dtype"] = torch.bfloat16
    with pytest.raises(ValueError):
        tc.matmul(a, b, **kw)


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")
def test_host_output_or_workspace_rejected():
    a = torch.zeros((256, 64), dtype=torch.float16, device="cuda")
    b = torch.zeros((64, 256), dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        tc.matmul(a, b, out=torch.empty((256, 256), dtype=torch.float16))
    with pytest.raises(ValueError):
        tc.matmul(a, b, workspace=torch.zeros(1 << 20, dtype=torch.uint8))
    with pytest.raises(ValueError):
        tc.matmul_acc(a, b, torch.zeros((256, 256), dtype=torch.float16))
    x = torch.zeros((32, 256), device="cuda")
    with pytest.raises(ValueError):
        tc.add_matrices(x, x, out=torch.empty((32, 256)))
    # nothing was launched: the device is clean and a valid call still works
    c = tc.matmul(a, b)
    torch.cuda.synchronize()
    assert torch.count_nonzero(c).item() == 0
