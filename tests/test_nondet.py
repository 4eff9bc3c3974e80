"""The non-deterministic weight gradient (the MoE grouped GEMM pull request's non-deterministic
package, "Mode rules"): only the row chunks of the split form are added in an unordered way
(fp32 atomic adds into the result); everything else is the deterministic kernel.

CPU: the C entry refuses any deterministic value but 0 and the usual bad arguments before
anything is launched; the binding takes deterministic keyword-only and runs only for the bool
False.  GPU: results against the fp64 oracle (fp32 and bf16, overwrite and accumulate, several
splits, empty and one-row groups), the unsplit form bitwise equal to grouped_det_gemm_wgrad, and
PyTorch's deterministic-mode alert raised before an order-varying launch only."""
import ctypes
import os
import warnings

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_bf16_close, assert_bitwise, assert_fp32_close, inputs_on, to64

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "moe_ragged_bf16_grouped_b300", "libgdg.so")
EINVAL, EWORKSPACE = 1, 4
A, B, OUT, OFFS = 0x100000, 0x40000000, 0x80000000, 0xC0000000


class Args(ctypes.Structure):
    _fields_ = [("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("rows", ctypes.c_int64), ("offs_kind", ctypes.c_int32),
                ("split_rows", ctypes.c_int32),
                ("out_ld", ctypes.c_int64), ("out_es", ctypes.c_int64)]


def _c():
    lib = ctypes.CDLL(LIB)
    f = lib.grouped_gemm_wgrad
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(Args), ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    w = lib.grouped_gemm_wgrad_workspace_bytes
    w.restype = ctypes.c_size_t
    w.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int32]
    return f, w


def test_c_entry_refusals_before_launch():
    f, w = _c()
    args = Args(A, B, OUT, None, 0, 512, 0, 64)
    for det in (1, -1, 2):
        assert f(ctypes.byref(args), OFFS, 4, 256, 256, 1, 0, det, None) == EINVAL
    assert f(None, OFFS, 4, 256, 256, 1, 0, 0, None) == EINVAL
    assert f(ctypes.byref(Args(A, B, OUT, None, 0, 512, 0, 100)), OFFS, 4, 256, 256, 1, 0, 0,
             None) == EINVAL                                        # split not a multiple of 64
    # a bf16 out in the split form needs the fp32 sums' workspace
    assert f(ctypes.byref(args), OFFS, 4, 256, 256, 0, 0, 0, None) == EWORKSPACE
    assert w(512, 4, 256, 256, 0, 0, 64) == 4 * 256 * 256 * 4
    assert w(512, 4, 256, 256, 1, 0, 64) == 0                       # fp32: adds go into out
    assert w(512, 4, 256, 256, 0, 0, -1) == 0                       # unsplit: no workspace
    assert w(512, 4, 250, 256, 0, 0, 64) == ctypes.c_size_t(-1).value


def test_binding_mode_rule():
    import moe_ragged_bf16_grouped_b300 as gdg
    g = torch.zeros((4, 8), dtype=torch.bfloat16)
    for bad in (True, None, 0, 1, "False", np.False_):
        with pytest.raises(ValueError, match="deterministic=False"):
            gdg.grouped_gemm_wgrad(g, g, torch.zeros(1, dtype=torch.int32), deterministic=bad)
    with pytest.raises(ValueError, match="deterministic=False"):
        gdg.grouped_gemm_wgrad(g, g, torch.zeros(1, dtype=torch.int32))   # omitted: the default


CASES = [
    # sizes, split_rows
    ([900, 0, 1, 333, 64, 2600, 17], 128),
    ([900, 0, 1, 333, 64, 2600, 17], 64),
    ([7000, 6500], 0),                 # the automatic split (few tiles, long groups)
    ([3000, 5, 0, 2500], 2304),        # chunks longer than 2048 rows (fp32 chunking inside)
]


@pytest.mark.gpu
@pytest.mark.parametrize("sizes,split", CASES)
def test_against_the_oracle(cuda_lib, sizes, split):
    w = wl.Workload("nd", E=len(sizes), N=512, K=384, ops=(), main_grad_std=1.0)
    h, d = inputs_on(w, "cuda", seed=12, sizes=sizes)
    ref = oracle.wgrad(h["G"], h["X"], h["offs_np"], w.E)
    empty = torch.from_numpy(np.array(sizes) == 0).to("cuda")
    assert cuda_lib.grouped_det_gemm_auto_split_rows(h["rows"], w.E, w.N, w.K) > 0 or split > 0
    dw = cuda_lib.grouped_gemm_wgrad(d["G"], d["X"], d["offs"], out_dtype=torch.float32,
                                     split_rows=split, deterministic=False)
    assert_fp32_close(dw, ref, "fp32 overwrite")
    assert torch.all(dw[empty].view(torch.int32) == 0), "empty group must give +0.0"
    acc = d["main_grad"].clone()
    cuda_lib.grouped_gemm_wgrad(d["G"], d["X"], d["offs"], out=acc, accumulate=True,
                                split_rows=split, deterministic=False)
    assert_fp32_close(acc, h["main_grad"].double().numpy() + ref, "fp32 accumulate")
    assert torch.equal(acc[empty].view(torch.int32), d["main_grad"][empty].view(torch.int32))
    dw16 = cuda_lib.grouped_gemm_wgrad(d["G"], d["X"], d["offs"], split_rows=split,
                                       deterministic=False)
    assert_bf16_close(dw16, ref, "bf16 overwrite")
    mg16 = d["main_grad"].to(torch.bfloat16)
    acc16 = mg16.clone()
    cuda_lib.grouped_gemm_wgrad(d["G"], d["X"], d["offs"], out=acc16, accumulate=True,
                                split_rows=split, deterministic=False)
    assert_bf16_close(acc16, to64(mg16) + ref, "bf16 accumulate")
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0


@pytest.mark.gpu
def test_unsplit_form_is_the_deterministic_kernel(cuda_lib):
    w = wl.Workload("nd_unsplit", E=5, N=512, K=320, ops=(), main_grad_std=1.0)
    _, d = inputs_on(w, "cuda", seed=13, sizes=[300, 0, 1, 2200, 17])
    for dt in (torch.float32, torch.bfloat16):
        nd = cuda_lib.grouped_gemm_wgrad(d["G"], d["X"], d["offs"], out_dtype=dt, split_rows=-1,
                                         deterministic=False)
        det = cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out_dtype=dt,
                                              split_rows=-1)
        assert_bitwise(nd, det, f"unsplit {dt}")


@pytest.mark.gpu
def test_deterministic_mode_alerts_before_order_varying_launches_only(cuda_lib):
    w = wl.Workload("nd_alert", E=2, N=256, K=256, ops=(), main_grad_std=1.0)
    _, d = inputs_on(w, "cuda", seed=14, sizes=[700, 500])
    out = torch.full((2, 256, 256), 7.0, dtype=torch.float32, device="cuda")
    prev = torch.are_deterministic_algorithms_enabled()
    prev_warn = torch.is_deterministic_algorithms_warn_only_enabled()
    try:
        torch.use_deterministic_algorithms(True)
        with pytest.raises(RuntimeError, match="grouped_det_gemm_wgrad"):
            cuda_lib.grouped_gemm_wgrad(d["G"], d["X"], d["offs"], out=out, split_rows=128,
                                        deterministic=False)
        torch.cuda.synchronize()
        assert torch.all(out == 7.0), "the refused call must launch nothing"
        # the unsplit form runs in a fixed order: no alert
        cuda_lib.grouped_gemm_wgrad(d["G"], d["X"], d["offs"], out=out, split_rows=-1,
                                    deterministic=False)
        torch.use_deterministic_algorithms(True, warn_only=True)
        with warnings.catch_warnings(record=True) as rec:
            warnings.simplefilter("always")
            cuda_lib.grouped_gemm_wgrad(d["G"], d["X"], d["offs"], out=out, split_rows=128,
                                        deterministic=False)
        assert any("grouped_det_gemm_wgrad" in str(r.message) for r in rec)
    finally:
        torch.use_deterministic_algorithms(prev, warn_only=prev_warn)
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0
