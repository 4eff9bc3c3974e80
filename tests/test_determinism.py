"""Bitwise run-to-run reproducibility (10 launches) of every operation and form."""
import pytest
import torch

import workloads as wl
from helpers import assert_bitwise, inputs_on

pytestmark = pytest.mark.gpu

DEV = "cuda"


def test_ten_runs_bitwise(cuda_lib):
    w = wl.Workload("det", E=7, N=512, K=384, ops=(), main_grad_std=0.01)
    h, d = inputs_on(w, DEV, seed=5, sizes=[900, 0, 1, 333, 64, 2600, 17])
    runs = {k: [] for k in ("fwd", "dgrad", "w16", "w32", "split", "acc")}
    for _ in range(10):
        runs["fwd"].append(cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], d["offs"]))
        runs["dgrad"].append(cuda_lib.grouped_det_gemm_dgrad(d["G"], d["W"], d["offs"]))
        runs["w16"].append(cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"],
                                                           split_rows=-1))
        runs["w32"].append(cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"],
                                                           out_dtype=torch.float32, split_rows=-1))
        runs["split"].append(cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"],
                                                             out_dtype=torch.float32,
                                                             split_rows=192))
        acc = d["main_grad"].clone()
        cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=acc, accumulate=True,
                                        split_rows=-1)
        runs["acc"].append(acc)
    for k, rs in runs.items():
        for r in rs[1:]:
            assert_bitwise(r, rs[0], k)
