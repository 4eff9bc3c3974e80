"""The weight-gradient entry point that allocates nothing.

Some callers cannot call cudaMalloc where they need a weight gradient (code inside a
memory pool or allocator, runtimes that hand out only the step's tensors).  For them
grouped_det_gemm_wgrad_noalloc runs the split form with the library's own fixed device
scratch instead of a caller workspace.  These tests call it through the C ABI and compare
it with grouped_det_gemm_wgrad given a caller workspace and the same split_rows.  This
file is collected last so that a run stopping at the first failure has run every other
test first.
"""
import ctypes
import os

import pytest
import torch

import workloads as wl
from helpers import assert_bitwise, assert_fp32_close, inputs_on, to64

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "moe_ragged_bf16_grouped_b300", "libgdg.so")
EINVAL, EWORKSPACE = 1, 4


class Args(ctypes.Structure):
    _fields_ = [("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("rows", ctypes.c_int64), ("offs_kind", ctypes.c_int32),
                ("split_rows", ctypes.c_int32),
                ("out_ld", ctypes.c_int64), ("out_es", ctypes.c_int64)]


def _fn():
    f = ctypes.CDLL(LIB).grouped_det_gemm_wgrad_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(Args), ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    return f


def noalloc_split_rows(rows, E, N, K, auto):
    """What split_rows = 0 resolves to: the automatic value if its partial tiles fit in the
    fixed scratch (at most 64 tiles of 256 x 256 fp32), else the smallest multiple of 64 whose
    tiles fit; None when nothing fits."""
    tpe = -(-N // 256) * -(-K // 256)
    chunks = 64 // tpe - E
    if chunks < 1:
        return None
    if auto > 0 and -(-rows // auto) <= chunks:
        return auto
    return -(-(-(-max(rows, 1) // chunks)) // 64) * 64


def test_refuses_before_any_launch():
    """Refusals happen on the host: no device is touched (fake, aligned addresses)."""
    f = _fn()
    # 1M rows cut into 64-row chunks need far more than the fixed scratch
    big = Args(0x100000, 0x40000000, 0x80000000, None, 0, 1 << 20, 0, 64)
    assert f(ctypes.byref(big), 0xC0000000, 64, 4096, 4096, 1, 0, None) == EWORKSPACE
    # split_rows = 0 with shapes whose partials cannot fit even one chunk per group
    # (16 tiles per expert x (4 experts + 1 chunk) > 64 tiles)
    auto0 = Args(0x100000, 0x40000000, 0x80000000, None, 0, 4096, 0, 0)
    assert f(ctypes.byref(auto0), 0xC0000000, 4, 1024, 1024, 1, 0, None) == EWORKSPACE
    neg = Args(0x100000, 0x40000000, 0x80000000, None, 0, 512, 0, -1)
    assert f(ctypes.byref(neg), 0xC0000000, 4, 256, 256, 1, 0, None) == EINVAL
    assert f(None, 0xC0000000, 4, 256, 256, 1, 0, None) == EINVAL


def _call(f, g, x, offs, out, split_rows, accumulate, kind):
    a = Args(g.data_ptr(), x.data_ptr(), out.data_ptr(), None, 0, g.shape[0], kind, split_rows)
    stream = torch.cuda.current_stream().cuda_stream
    st = f(ctypes.byref(a), offs.data_ptr(), offs.numel() - kind, g.shape[1], x.shape[1],
           1 if out.dtype == torch.float32 else 0, int(accumulate), stream)
    assert st == 0, st


@pytest.mark.gpu
def test_matches_workspace_entry_point_on_two_calls(cuda_lib):
    f = _fn()
    cases = [
        # (workload, sizes, kind, split_rows, accumulate, out dtype)
        (wl.Workload("r", E=6, N=512, K=320, ops=(), main_grad_std=1.0),
         [300, 0, 1, 17, 513, 255], wl.OFFS_ENDS, 128, False, torch.float32),
        (wl.Workload("t", E=4, N=256, K=256, ops=(), main_grad_std=1.0),
         [200, 0, 311, 1], wl.OFFS_INDPTR, 0, True, torch.float32),
        # split_rows = 0 where the automatic split's partials do not fit: a coarser split
        # that fits is chosen (65536 rows, 1 tile per expert: 1152-row chunks, 61 tiles)
        (wl.Workload("big", E=4, N=256, K=256, ops=(), main_grad_std=1.0),
         [30000, 0, 35535, 1], wl.OFFS_ENDS, 0, False, torch.bfloat16),
    ]
    for w, sizes, kind, split, acc, dt in cases:     # two calls in a row, different shapes
        _, d = inputs_on(w, "cuda", seed=7, sizes=sizes, kind=kind)
        resolved0 = split if split > 0 else noalloc_split_rows(
            d["rows"], w.E, w.N, w.K,
            cuda_lib.grouped_det_gemm_auto_split_rows(d["rows"], w.E, w.N, w.K))
        need = cuda_lib.grouped_det_gemm_workspace_bytes(
            cuda_lib.GDG_OP_WGRAD, d["rows"], w.E, w.N, w.K, dt, acc, resolved0)
        assert 0 < need <= cuda_lib.GDG_NOALLOC_SCRATCH_BYTES
        start = d["main_grad"].to(dt) if acc else torch.full((w.E, w.N, w.K), 9.0,
                                                              dtype=dt, device="cuda")
        resolved = split if split > 0 else noalloc_split_rows(
            d["rows"], w.E, w.N, w.K,
            cuda_lib.grouped_det_gemm_auto_split_rows(d["rows"], w.E, w.N, w.K))
        ref = cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=start.clone(),
                                              accumulate=acc, split_rows=resolved,
                                              offs_kind=kind)
        got = start.clone()
        _call(f, d["G"], d["X"], d["offs"], got, split, acc, kind)
        torch.cuda.synchronize()
        assert cuda_lib.gdg_device_error() == 0
        if dt == torch.float32:
            assert_fp32_close(got, to64(ref), "no-alloc vs workspace entry point")
        assert_bitwise(got, ref, f"no-alloc vs workspace entry point (split_rows {resolved})")
