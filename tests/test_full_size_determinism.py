"""Bitwise run-to-run reproducibility over 10 launches at full size: every large workload, seed 0,
through the calls bench.py times (the MoE grouped GEMM pull request's test list: run to run over
10 launches; the wgrad-heavy workload asks for it explicitly).

* Mixtral-style and fine-grained: fwd, dgrad and wgrad with bf16 dW;
* wgrad-heavy: wgrad with fp32 accumulate into a fresh copy of main_grad on every run (the
  2048-row fp32 chunking of long groups runs here);
* decode-sized: fwd and dgrad.

Each run's output is compared bit for bit with the first run's on the device.
"""
import pytest
import torch

import workloads as wl
from helpers import assert_bitwise

pytestmark = pytest.mark.gpu

DEV = "cuda"
RUNS = 10


def _ops(cuda_lib, w, d):
    ops = {}
    if "fwd" in w.ops:
        Y = torch.empty((d["rows"], w.N), dtype=torch.bfloat16, device=DEV)
        dX = torch.empty((d["rows"], w.K), dtype=torch.bfloat16, device=DEV)
        ops["fwd"] = lambda: cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], d["offs"], out=Y)
        ops["dgrad"] = lambda: cuda_lib.grouped_det_gemm_dgrad(d["G"], d["W"], d["offs"], out=dX)
    if "wgrad_bf16" in w.ops:
        dW = torch.empty((w.E, w.N, w.K), dtype=torch.bfloat16, device=DEV)
        ops["wgrad"] = lambda: cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=dW)
    if "wgrad_fp32_acc" in w.ops:
        acc = torch.empty_like(d["main_grad"])

        def wgrad_acc():
            acc.copy_(d["main_grad"])
            return cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=acc,
                                                   accumulate=True)
        ops["wgrad_fp32_acc"] = wgrad_acc
    return ops


@pytest.mark.parametrize("name", ["mixtral", "fine_grained", "wgrad_heavy", "decode"])
def test_ten_runs_bitwise_full_size(cuda_lib, name):
    w = wl.WORKLOADS[name]
    d = wl.make_inputs(w, seed=0, device=DEV)
    for op, fn in _ops(cuda_lib, w, d).items():
        first = fn().clone()
        for i in range(1, RUNS):
            assert_bitwise(fn(), first, f"{name} {op} run {i}")
        del first
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0
