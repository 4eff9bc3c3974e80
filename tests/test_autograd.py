"""The autograd wrapper on the GPU with the library's kernels: gradients bitwise equal to the
direct calls, the fused main_grad accumulation bitwise equal to main_grad.add_(dW) (fp32 and bf16
main_grad), repeated backwards adding again, and the placeholder of the Megatron convention."""
import pytest
import torch

import workloads as wl
from helpers import assert_bitwise, inputs_on

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _case():
    w = wl.Workload("ag", E=4, N=512, K=384, ops=(), main_grad_std=0.01)
    d = inputs_on(w, DEV, seed=8, sizes=[700, 0, 1, 2300])[1]
    dy = wl.normal_bf16((d["rows"], w.N), 1.0, 8, 9, DEV)
    return d, dy


def test_gradients_match_direct_calls(cuda_lib):
    d, dy = _case()
    x = d["X"].clone().requires_grad_()
    w = d["W"].clone().requires_grad_()
    y = cuda_lib.grouped_det_mm(x, w, d["offs"])
    assert_bitwise(y.detach(), cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], d["offs"]), "Y")
    y.backward(dy)
    assert_bitwise(x.grad, cuda_lib.grouped_det_gemm_dgrad(dy, d["W"], d["offs"]), "x.grad")
    assert_bitwise(w.grad, cuda_lib.grouped_det_gemm_wgrad(dy, d["X"], d["offs"]), "w.grad")


@pytest.mark.parametrize("mg_dtype", [torch.float32, torch.bfloat16])
def test_fused_main_grad(cuda_lib, mg_dtype):
    d, dy = _case()
    x = d["X"].clone().requires_grad_()
    w = d["W"].clone().requires_grad_()
    mg0 = d["main_grad"].to(mg_dtype)
    w.main_grad = mg0.clone()
    w.grad_added_to_main_grad = False
    y = cuda_lib.grouped_det_mm(x, w, d["offs"], fuse_wgrad_accumulation=True)
    y.backward(dy, retain_graph=True)
    y.backward(dy)                                  # every backward adds again
    dw = cuda_lib.grouped_det_gemm_wgrad(dy, d["X"], d["offs"], out_dtype=mg_dtype)
    assert_bitwise(w.main_grad, mg0.clone().add_(dw).add_(dw), "main_grad")
    assert w.grad_added_to_main_grad is True and w.grad.shape == w.shape
    assert_bitwise(x.grad, cuda_lib.grouped_det_gemm_dgrad(dy, d["W"], d["offs"]) * 2, "x.grad")
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0
