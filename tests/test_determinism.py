"""Bitwise run-to-run reproducibility (10 launches) of every operation and form, and bitwise
independence from the persistent grid size (the unit -> pair assignment changes, each unit's
arithmetic does not)."""
import ctypes

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


def test_bitwise_across_grid_sizes(cuda_lib):
    w = wl.Workload("det_grid", E=7, N=512, K=384, ops=(), main_grad_std=0.01)
    h, d = inputs_on(w, DEV, seed=6, sizes=[900, 0, 1, 333, 64, 2600, 17])
    setcap = cuda_lib._lib.gdg_test_set_max_pairs
    setcap.restype = None
    setcap.argtypes = [ctypes.c_int]

    def all_ops():
        acc = d["main_grad"].clone()
        cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=acc, accumulate=True,
                                        split_rows=-1)
        return {
            "fwd": cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], d["offs"]),
            "dgrad": cuda_lib.grouped_det_gemm_dgrad(d["G"], d["W"], d["offs"]),
            "w16": cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], split_rows=-1),
            "w32": cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"],
                                                   out_dtype=torch.float32, split_rows=-1),
            "split": cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"],
                                                     out_dtype=torch.float32, split_rows=192),
            "acc": acc,
        }

    full = all_ops()
    try:
        for cap in (1, 3, 13):
            setcap(cap)
            got = all_ops()
            for k in full:
                assert_bitwise(got[k], full[k], f"{k} with {cap} pairs")
    finally:
        setcap(0)
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0
