"""The autograd wrapper on the GPU with the library's kernels: Y, x.grad and w.grad against the
fp64 oracle (docs page "Autograd": the backward is dgrad for x and wgrad for w) and bitwise equal
to the direct calls; the fused main_grad accumulation (MoE grouped GEMM pull request,
"Deterministic weight-gradient accumulation") against main_grad + 2 dW from the oracle after two
backwards, and bitwise equal to main_grad.add_(dW) twice (fp32 and bf16 main_grad); the
placeholder of the Megatron convention."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_bf16_close, assert_bitwise, assert_fp32_close, inputs_on, to64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _case():
    w = wl.Workload("ag", E=4, N=512, K=384, ops=(), main_grad_std=0.01)
    h, d = inputs_on(w, DEV, seed=8, sizes=[700, 0, 1, 2300])
    dy = wl.normal_bf16((d["rows"], w.N), 1.0, 8, 9, DEV)
    return h, d, dy


def test_gradients_match_oracle_and_direct_calls(cuda_lib):
    h, d, dy = _case()
    x = d["X"].clone().requires_grad_()
    w = d["W"].clone().requires_grad_()
    y = cuda_lib.grouped_det_mm(x, w, d["offs"])
    y.backward(dy)
    dy_h = dy.cpu()
    assert_bf16_close(y.detach(), oracle.fwd(h["X"], h["W"], h["offs_np"]), "Y vs oracle")
    assert_bf16_close(x.grad, oracle.dgrad(dy_h, h["W"], h["offs_np"]), "x.grad vs oracle")
    assert_bf16_close(w.grad, oracle.wgrad(dy_h, h["X"], h["offs_np"], 4), "w.grad vs oracle")
    assert_bitwise(y.detach(), cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], d["offs"]), "Y")
    assert_bitwise(x.grad, cuda_lib.grouped_det_gemm_dgrad(dy, d["W"], d["offs"]), "x.grad")
    assert_bitwise(w.grad, cuda_lib.grouped_det_gemm_wgrad(dy, d["X"], d["offs"]), "w.grad")


@pytest.mark.parametrize("mg_dtype", [torch.float32, torch.bfloat16])
def test_fused_main_grad(cuda_lib, mg_dtype):
    h, d, dy = _case()
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
    # Against the oracle: main_grad0 + 2 dW (two backwards, each adding once).
    ref = to64(mg0) + 2.0 * oracle.wgrad(dy.cpu(), h["X"], h["offs_np"], 4)
    if mg_dtype == torch.float32:
        assert_fp32_close(w.main_grad, ref, "main_grad vs oracle")
    else:
        assert_bf16_close(w.main_grad, ref, "bf16 main_grad vs oracle")
    assert np.all(to64(w.main_grad)[1] == to64(mg0)[1] + 0.0), "empty group changed main_grad"
    assert w.grad_added_to_main_grad is True and w.grad.shape == w.shape
    assert_bitwise(x.grad, cuda_lib.grouped_det_gemm_dgrad(dy, d["W"], d["offs"]) * 2, "x.grad")
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0
