"""GPU tests of strided outputs (unit stride along the last dimension): Y / dX written into
column slices of wider buffers, dW into a permuted [N, E, K] buffer, and the fused accumulate into
a main_grad that is a column slice of a wider parameter buffer (the accumulate contract of the MoE
grouped GEMM pull request allows such views).

Strided results must equal the dense call's bit for bit (the kernels compute the same values;
only the addresses change), and every byte of the wider buffer outside the view must keep its
sentinel.
"""
import pytest
import torch

import workloads as wl
from helpers import assert_bitwise, inputs_on

pytestmark = pytest.mark.gpu

DEV = "cuda"

CASES = [
    # name, E, N, K, sizes, lead, pad, kind
    ("dense_tiles", 3, 256, 320, [300, 0, 77], 0, 2, wl.OFFS_ENDS),
    ("odd_shape", 2, 136, 200, [129, 40], 1, 0, wl.OFFS_INDPTR),
]


def case(spec, seed=9):
    name, E, N, K, sizes, lead, pad, kind = spec
    w = wl.Workload(name, E=E, N=N, K=K, ops=(), main_grad_std=1.0)
    return inputs_on(w, DEV, seed=seed, sizes=sizes, kind=kind, pad_rows=pad, lead=lead)


def bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


@pytest.mark.parametrize("spec", CASES, ids=[c[0] for c in CASES])
def test_fwd_dgrad_into_column_slices(cuda_lib, spec):
    h, d = case(spec)
    w, kind, rows = h["workload"], h["kind"], h["rows"]
    for fn, a, cols in ((cuda_lib.grouped_det_gemm_fwd, d["X"], w.N),
                        (cuda_lib.grouped_det_gemm_dgrad, d["G"], w.K)):
        dense = fn(a, d["W"], d["offs"], out=torch.full((rows, cols), -7.0, dtype=torch.bfloat16,
                                                       device=DEV), offs_kind=kind)
        wide = torch.full((rows, cols + 40), -5.0, dtype=torch.bfloat16, device=DEV)
        view = wide[:, 16:16 + cols]              # row stride cols + 40, 32-byte offset
        view.fill_(-7.0)
        fn(a, d["W"], d["offs"], out=view, offs_kind=kind)
        assert_bitwise(view, dense, f"{fn.__name__} strided")
        assert torch.all(wide[:, :16] == -5.0) and torch.all(wide[:, 16 + cols:] == -5.0), \
            f"{fn.__name__} wrote outside its view"
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0


@pytest.mark.parametrize("split_rows", [-1, 64])
@pytest.mark.parametrize("spec", CASES, ids=[c[0] for c in CASES])
def test_wgrad_into_permuted_buffer(cuda_lib, spec, split_rows):
    """dW[e] rows interleaved by expert: out = buf[N, E, K].permute(1, 0, 2)."""
    h, d = case(spec)
    w, kind = h["workload"], h["kind"]
    for dtype in (torch.float32, torch.bfloat16):
        dense = cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out_dtype=dtype,
                                                split_rows=split_rows, offs_kind=kind)
        buf = torch.full((w.N, w.E, w.K), 3.0, dtype=dtype, device=DEV)
        out = buf.permute(1, 0, 2)
        cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=out,
                                        split_rows=split_rows, offs_kind=kind)
        assert_bitwise(out, dense, f"wgrad {dtype} permuted")
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0


@pytest.mark.parametrize("split_rows", [-1, 64])
@pytest.mark.parametrize("spec", CASES, ids=[c[0] for c in CASES])
def test_accumulate_into_strided_main_grad(cuda_lib, spec, split_rows):
    """main_grad = param_buffer[:, :, 8:8 + K]: the fused add equals main_grad.add_(dW) bitwise
    and the buffer's other columns keep their bits."""
    h, d = case(spec)
    w, kind = h["workload"], h["kind"]
    for dtype in (torch.float32, torch.bfloat16):
        dW = cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out_dtype=dtype,
                                             split_rows=split_rows, offs_kind=kind)
        big = torch.full((w.E, w.N, w.K + 24), 11.0, dtype=dtype, device=DEV)
        mg = big[:, :, 8:8 + w.K]
        mg.copy_(d["main_grad"].to(dtype))
        before = big.clone()
        expect = mg.clone().add_(dW)
        cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=mg, accumulate=True,
                                        split_rows=split_rows, offs_kind=kind)
        assert_bitwise(mg, expect, f"strided accumulate {dtype}")
        assert torch.equal(bits(big[:, :, :8]), bits(before[:, :, :8]))
        assert torch.equal(bits(big[:, :, 8 + w.K:]), bits(before[:, :, 8 + w.K:]))
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0


def test_autograd_fused_into_strided_main_grad(cuda_lib):
    """grouped_det_mm with fuse_wgrad_accumulation and w.main_grad a strided view."""
    h, d = case(CASES[0])
    w = h["workload"]
    x = d["X"].clone().requires_grad_(True)
    wt = d["W"].clone().requires_grad_(True)
    big = torch.zeros((w.E, w.N, w.K + 8), dtype=torch.float32, device=DEV)
    wt.main_grad = big[:, :, :w.K]
    wt.main_grad.copy_(d["main_grad"])
    expect = wt.main_grad.clone().add_(
        cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out_dtype=torch.float32))
    y = cuda_lib.grouped_det_mm(x, wt, d["offs"], fuse_wgrad_accumulation=True)
    y.backward(d["G"])
    assert_bitwise(wt.main_grad, expect, "autograd strided main_grad")
    assert torch.all(big[:, :, w.K:] == 0)
