"""GPU parity at the library's limits: the largest expert count the C ABI takes
(GDG_MAX_EXPERTS = 1024), with mostly empty and 1-3-row groups plus a few longer ones, through
every op and both wgrad forms (the split form's ordered reduce keeps per-expert tables of that
size in shared memory), in both offset conventions."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import (assert_bf16_close, assert_fp32_close, group_rows_mask, inputs_on)

pytestmark = pytest.mark.gpu

DEV = "cuda"
E_MAX = 1024


def limit_sizes():
    rng = np.random.default_rng(21)
    sizes = rng.choice([0, 0, 0, 1, 2, 3], size=E_MAX).astype(int)
    sizes[[5, 600, 1023]] = [17, 300, 33]     # a few longer groups, the last expert included
    sizes[0] = 0
    return [int(v) for v in sizes]


@pytest.mark.parametrize("kind", [wl.OFFS_ENDS, wl.OFFS_INDPTR], ids=["ends", "indptr"])
def test_max_experts(cuda_lib, kind):
    w = wl.Workload("max_experts", E=E_MAX, N=256, K=128, ops=(), main_grad_std=1.0)
    h, d = inputs_on(w, DEV, seed=3, sizes=limit_sizes(), kind=kind, pad_rows=2,
                     lead=1 if kind == wl.OFFS_INDPTR else 0)
    rows = h["rows"]
    mask = group_rows_mask(h["offs_np"], kind, E_MAX, rows)
    tmask = torch.from_numpy(mask).to(DEV)
    Y = cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], d["offs"], offs_kind=kind)
    assert_bf16_close(Y[tmask], oracle.fwd(h["X"], h["W"], h["offs_np"], kind)[mask], "fwd")
    dX = cuda_lib.grouped_det_gemm_dgrad(d["G"], d["W"], d["offs"], offs_kind=kind)
    assert_bf16_close(dX[tmask], oracle.dgrad(h["G"], h["W"], h["offs_np"], kind)[mask], "dgrad")
    ref = oracle.wgrad(h["G"], h["X"], h["offs_np"], E_MAX, kind)
    for split in (-1, 64):
        dW = cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out_dtype=torch.float32,
                                             split_rows=split, offs_kind=kind)
        assert_fp32_close(dW, ref, f"wgrad split={split}")
        empty = torch.from_numpy(np.array(h["sizes"]) == 0).to(DEV)
        assert torch.all(dW[empty].view(torch.int32) == 0), "empty groups must give +0.0"
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0
