"""Prepared launches and CUDA graphs (docs page, "Prepared launches"; the accumulate notes of
the MoE grouped GEMM pull request: every launch and every graph replay adds again).

A plan binds the checks, tensor maps and grid once; its launches must give the direct call's
bits.  Captured in a CUDA graph, plans and direct calls replay with the offsets read on the GPU:
new offsets written into the bound buffer are honoured, and accumulate adds on every replay."""
import pytest
import torch

import oracle
import workloads as wl
from helpers import (assert_bf16_close, assert_bitwise, assert_fp32_close, group_rows_mask,
                     inputs_on, to64)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _case(sizes, seed=3, host=False):
    w = wl.Workload("graph", E=len(sizes), N=512, K=320, ops=(), main_grad_std=1.0)
    h, d = inputs_on(w, DEV, seed=seed, sizes=sizes)
    return (h, d) if host else d


def test_plan_launch_matches_direct_call(cuda_lib):
    d = _case([300, 0, 1, 2200, 17])
    G, X, W, offs, mg = d["G"], d["X"], d["W"], d["offs"], d["main_grad"]
    pf = cuda_lib.prepare_grouped_det_gemm_fwd(X, W, offs)
    pd = cuda_lib.prepare_grouped_det_gemm_dgrad(G, W, offs)
    pw = cuda_lib.prepare_grouped_det_gemm_wgrad(G, X, offs)
    ps = cuda_lib.prepare_grouped_det_gemm_wgrad(G, X, offs, out_dtype=torch.float32,
                                                 split_rows=256)
    acc = mg.clone()
    pa = cuda_lib.prepare_grouped_det_gemm_wgrad(G, X, offs, out=acc, accumulate=True)
    for _ in range(2):
        pf.launch(), pd.launch(), pw.launch(), ps.launch()
    pa.launch()
    h = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    assert_bf16_close(pf.out, oracle.fwd(h["X"], h["W"], h["offs_np"]), "fwd plan vs oracle")
    assert_bf16_close(pd.out, oracle.dgrad(h["G"], h["W"], h["offs_np"]), "dgrad plan vs oracle")
    ref_dw = oracle.wgrad(h["G"], h["X"], h["offs_np"], 5)
    assert_bf16_close(pw.out, ref_dw, "wgrad plan vs oracle")
    assert_fp32_close(ps.out, ref_dw, "split plan vs oracle")
    assert_fp32_close(acc, to64(mg) + ref_dw, "accumulate plan vs oracle")
    assert_bitwise(pf.out, cuda_lib.grouped_det_gemm_fwd(X, W, offs), "fwd plan")
    assert_bitwise(pd.out, cuda_lib.grouped_det_gemm_dgrad(G, W, offs), "dgrad plan")
    assert_bitwise(pw.out, cuda_lib.grouped_det_gemm_wgrad(G, X, offs), "wgrad plan")
    assert_bitwise(ps.out, cuda_lib.grouped_det_gemm_wgrad(G, X, offs, out_dtype=torch.float32,
                                                           split_rows=256), "split plan")
    dw32 = cuda_lib.grouped_det_gemm_wgrad(G, X, offs, out_dtype=torch.float32)
    assert_bitwise(acc, mg.clone().add_(dw32), "accumulate plan")
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0


def test_graph_replay_honours_new_offsets_and_adds_again(cuda_lib):
    sizes_a, sizes_b = [300, 0, 1, 2200, 17], [1000, 500, 0, 1, 1017]   # same rows
    h, d = _case(sizes_a, host=True)
    G, X, W, offs, mg = d["G"], d["X"], d["W"], d["offs"], d["main_grad"]
    offs_b = torch.from_numpy(wl.offsets(sizes_b)).to(DEV)
    acc = mg.clone()
    plans = [cuda_lib.prepare_grouped_det_gemm_fwd(X, W, offs),
             cuda_lib.prepare_grouped_det_gemm_wgrad(G, X, offs, out=acc, accumulate=True)]
    dX = torch.empty_like(X)
    dW = torch.empty((W.shape[0], W.shape[1], W.shape[2]), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm-up outside the capture (device set-up happens once)
        for pl in plans:
            pl.launch()
        cuda_lib.grouped_det_gemm_dgrad(G, W, offs, out=dX)
        cuda_lib.grouped_det_gemm_wgrad(G, X, offs, out=dW)
    torch.cuda.synchronize()
    acc.copy_(mg)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for pl in plans:
            pl.launch()
        cuda_lib.grouped_det_gemm_dgrad(G, W, offs, out=dX)
        cuda_lib.grouped_det_gemm_wgrad(G, X, offs, out=dW)
    torch.cuda.synchronize()
    assert torch.equal(acc, mg), "capture must not run the kernels"

    expect = mg.clone()
    expect64 = to64(mg)                    # main_grad + the oracle's dW of every replay so far
    rows, E = h["rows"], len(sizes_a)
    for sizes, o in ((sizes_a, None), (sizes_b, offs_b), (sizes_b, offs_b)):
        if o is not None:
            offs.copy_(o)                  # new offsets in the bound buffer
        g.replay()
        torch.cuda.synchronize()
        # Each replay against the oracle on the offsets it ran with.
        offs_np = wl.offsets(sizes)
        mask = group_rows_mask(offs_np, wl.OFFS_ENDS, E, rows)
        tmask = torch.from_numpy(mask).to(DEV)
        assert_bf16_close(plans[0].out[tmask], oracle.fwd(h["X"], h["W"], offs_np)[mask],
                          f"fwd replay {sizes} vs oracle")
        assert_bf16_close(dX[tmask], oracle.dgrad(h["G"], h["W"], offs_np)[mask],
                          f"dgrad replay {sizes} vs oracle")
        ref_dw = oracle.wgrad(h["G"], h["X"], offs_np, E)
        assert_bf16_close(dW, ref_dw, f"wgrad replay {sizes} vs oracle")
        expect64 = expect64 + ref_dw
        assert_fp32_close(acc, expect64, f"accumulate after replay {sizes} vs oracle")
        # ... and bitwise equal to the direct calls on the same offsets.
        dw32 = cuda_lib.grouped_det_gemm_wgrad(G, X, offs, out_dtype=torch.float32)
        expect.add_(dw32)                  # every replay adds again
        assert_bitwise(plans[0].out, cuda_lib.grouped_det_gemm_fwd(X, W, offs), f"fwd {sizes}")
        assert_bitwise(dX, cuda_lib.grouped_det_gemm_dgrad(G, W, offs), f"dgrad {sizes}")
        assert_bitwise(dW, cuda_lib.grouped_det_gemm_wgrad(G, X, offs), f"wgrad {sizes}")
        assert_bitwise(acc, expect, f"accumulate {sizes}")
    assert cuda_lib.gdg_device_error() == 0


def test_two_streams(cuda_lib):
    d1, d2 = _case([700, 3, 0, 400, 9], seed=4), _case([5, 600, 250, 0, 1], seed=5)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for s in (s1, s2):
        s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        y1 = cuda_lib.grouped_det_gemm_fwd(d1["X"], d1["W"], d1["offs"])
        w1 = cuda_lib.grouped_det_gemm_wgrad(d1["G"], d1["X"], d1["offs"])
    with torch.cuda.stream(s2):
        y2 = cuda_lib.grouped_det_gemm_fwd(d2["X"], d2["W"], d2["offs"])
        w2 = cuda_lib.grouped_det_gemm_wgrad(d2["G"], d2["X"], d2["offs"])
    torch.cuda.synchronize()
    assert_bitwise(y1, cuda_lib.grouped_det_gemm_fwd(d1["X"], d1["W"], d1["offs"]), "fwd s1")
    assert_bitwise(y2, cuda_lib.grouped_det_gemm_fwd(d2["X"], d2["W"], d2["offs"]), "fwd s2")
    assert_bitwise(w1, cuda_lib.grouped_det_gemm_wgrad(d1["G"], d1["X"], d1["offs"]), "wgrad s1")
    assert_bitwise(w2, cuda_lib.grouped_det_gemm_wgrad(d2["G"], d2["X"], d2["offs"]), "wgrad s2")
