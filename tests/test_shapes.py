"""GPU parity for shapes that are not multiples of the tiles: N % 256 != 0 and K % 64 != 0
(only N % 8 == K % 8 == 0 is required, for 16-byte aligned rows).

Every output lives inside a larger buffer whose bytes before and after it are a sentinel, so a
write past N or K (into the next expert's rows or past the end) is caught bitwise.  Cases mix
both fwd/dgrad row tiles (at most / more than 64 rows per group on average), both offset
conventions, empty and one-row groups, and N or K below one 64-wide block.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import (assert_bf16_close, assert_bitwise, assert_fp32_close, group_rows_mask,
                     inputs_on, to64)

pytestmark = pytest.mark.gpu

DEV = "cuda"
PAD = 64   # sentinel elements on each side of an output (64 * 2 or 4 bytes: keeps 16-byte alignment)

CASES = [
    # name, E, N, K, sizes, lead, pad, kind
    ("n136_k200", 3, 136, 200, [150, 0, 37], 0, 2, wl.OFFS_ENDS),
    ("n264_k328", 2, 264, 328, [300, 129], 1, 0, wl.OFFS_INDPTR),
    ("n8_k16", 2, 8, 16, [33, 5], 0, 0, wl.OFFS_ENDS),
    ("n520_k72", 4, 520, 72, [1, 700, 0, 64], 0, 3, wl.OFFS_ENDS),
    ("row_tile_128_n392_k456", 6, 392, 456, [3, 0, 5, 1, 17, 2], 0, 0, wl.OFFS_ENDS),
]


def case(spec, seed=5):
    name, E, N, K, sizes, lead, pad, kind = spec
    w = wl.Workload(name, E=E, N=N, K=K, ops=(), main_grad_std=1.0)
    return inputs_on(w, DEV, seed=seed, sizes=sizes, kind=kind, pad_rows=pad, lead=lead)


def fenced(shape, dtype, fill):
    """A tensor of `shape` inside a flat buffer with PAD sentinel elements on each side."""
    n = int(np.prod(shape))
    flat = torch.full((n + 2 * PAD,), fill, dtype=dtype, device=DEV)
    return flat, flat[PAD:PAD + n].view(shape)


def check_fence(flat, fill, what):
    head, tail = flat[:PAD], flat[-PAD:]
    ref = torch.full_like(head, fill)
    assert torch.equal(head.view(torch.int16 if flat.element_size() == 2 else torch.int32),
                       ref.view(torch.int16 if flat.element_size() == 2 else torch.int32)), \
        f"{what}: wrote before the output"
    assert torch.equal(tail.view(torch.int16 if flat.element_size() == 2 else torch.int32),
                       ref.view(torch.int16 if flat.element_size() == 2 else torch.int32)), \
        f"{what}: wrote past the output"


@pytest.mark.parametrize("spec", CASES, ids=[c[0] for c in CASES])
def test_fwd_dgrad_odd_shapes(cuda_lib, spec):
    h, d = case(spec)
    w, kind, rows = h["workload"], h["kind"], h["rows"]
    mask = group_rows_mask(h["offs_np"], kind, w.E, rows)
    tmask = torch.from_numpy(mask).to(DEV)
    flat, Y = fenced((rows, w.N), torch.bfloat16, -7.0)
    cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], d["offs"], out=Y, offs_kind=kind)
    assert_bf16_close(Y[tmask], oracle.fwd(h["X"], h["W"], h["offs_np"], kind)[mask], "fwd")
    assert torch.all(Y[~tmask] == -7.0), "fwd wrote rows outside groups"
    check_fence(flat, -7.0, "fwd")
    flat, dX = fenced((rows, w.K), torch.bfloat16, -7.0)
    cuda_lib.grouped_det_gemm_dgrad(d["G"], d["W"], d["offs"], out=dX, offs_kind=kind)
    assert_bf16_close(dX[tmask], oracle.dgrad(h["G"], h["W"], h["offs_np"], kind)[mask], "dgrad")
    assert torch.all(dX[~tmask] == -7.0), "dgrad wrote rows outside groups"
    check_fence(flat, -7.0, "dgrad")
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0


@pytest.mark.parametrize("split_rows", [-1, 64, 0])
@pytest.mark.parametrize("spec", CASES, ids=[c[0] for c in CASES])
def test_wgrad_odd_shapes(cuda_lib, spec, split_rows):
    h, d = case(spec)
    w, kind = h["workload"], h["kind"]
    ref = oracle.wgrad(h["G"], h["X"], h["offs_np"], w.E, kind)
    for dtype, close in ((torch.float32, assert_fp32_close), (torch.bfloat16, assert_bf16_close)):
        flat, dW = fenced((w.E, w.N, w.K), dtype, 3.0)
        cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=dW, split_rows=split_rows,
                                        offs_kind=kind)
        close(dW, ref, f"wgrad {dtype}")
        check_fence(flat, 3.0, f"wgrad {dtype}")
        for e in range(w.E):
            if h["sizes"][e] == 0:
                assert torch.all(dW[e] == 0) and not torch.any(torch.signbit(dW[e])), \
                    "empty group must give +0.0"
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0


@pytest.mark.parametrize("split_rows", [-1, 64])
@pytest.mark.parametrize("spec", CASES[:3], ids=[c[0] for c in CASES[:3]])
def test_wgrad_accumulate_odd_shapes(cuda_lib, spec, split_rows):
    """Fused accumulate == main_grad.add_(dW) bitwise, fp32 and bf16, and nothing outside."""
    h, d = case(spec)
    w, kind = h["workload"], h["kind"]
    for dtype in (torch.float32, torch.bfloat16):
        dW = cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out_dtype=dtype,
                                             split_rows=split_rows, offs_kind=kind)
        flat, mg = fenced((w.E, w.N, w.K), dtype, 5.0)
        mg.copy_(d["main_grad"].to(dtype))
        expect = mg.clone().add_(dW)
        cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=mg, accumulate=True,
                                        split_rows=split_rows, offs_kind=kind)
        assert_bitwise(mg, expect, f"accumulate {dtype}")
        check_fence(flat, 5.0, f"accumulate {dtype}")
    ref = oracle.wgrad_accumulate(d["main_grad"].cpu(), h["G"], h["X"], h["offs_np"], w.E, kind)
    mg = d["main_grad"].clone()
    cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=mg, accumulate=True,
                                    split_rows=split_rows, offs_kind=kind)
    assert_fp32_close(mg, ref, "fp32 accumulate vs oracle")


def test_integer_exact_odd_shape(cuda_lib):
    """Small-integer operands (every partial sum exact) on N=136, K=200: fwd, dgrad and wgrad
    equal the oracle bit for bit, so masking at the N and K edges is exact."""
    sizes = [37, 0, 130, 1]
    E, N, K = len(sizes), 136, 200
    rows = sum(sizes) + 2
    X = wl.integer_bf16((rows, K), -2, 2, seed=7, tag=1)
    G = wl.integer_bf16((rows, N), -2, 2, seed=7, tag=2)
    W = wl.integer_bf16((E, N, K), -1, 1, seed=7, tag=3)
    offs = wl.offsets(sizes)
    mask = group_rows_mask(offs, wl.OFFS_ENDS, E, rows)
    o = torch.from_numpy(offs).to(DEV)
    Y = cuda_lib.grouped_det_gemm_fwd(X.to(DEV), W.to(DEV), o)
    dX = cuda_lib.grouped_det_gemm_dgrad(G.to(DEV), W.to(DEV), o)
    yref, dref = oracle.fwd(X, W, offs), oracle.dgrad(G, W, offs)
    assert np.abs(yref[mask]).max() <= 256 and np.abs(dref[mask]).max() <= 256
    assert np.array_equal(to64(Y)[mask], yref[mask])
    assert np.array_equal(to64(dX)[mask], dref[mask])
    for split in (-1, 64):
        dW = cuda_lib.grouped_det_gemm_wgrad(G.to(DEV), X.to(DEV), o, out_dtype=torch.float32,
                                             split_rows=split)
        assert np.array_equal(to64(dW), oracle.wgrad(G, X, offs, E)), f"wgrad split={split}"
