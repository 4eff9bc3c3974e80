"""Failure detection on the GPU without a GPU fault.

The test-only entry point gdg_test_withhold_first_stage launches a normal call except that CTA
pair 0 arms its first pipeline stage and never fills it (a flag that nothing sets).  The pair's
bounded waits run out after about 2 s, it aborts cleanly and the library's device error word
reports GDG_ETIMEOUT; the host reads it after the launch.  The context must stay usable: the
same call without the hook then matches the oracle, with no error recorded.  No trap, device
assert, bad address or endless loop is involved.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_bf16_close, assert_fp32_close, group_rows_mask, inputs_on

pytestmark = pytest.mark.gpu

DEV = "cuda"
GDG_ETIMEOUT = 6


def withhold(gdg, op_code, args, dims, offs):
    f = gdg._lib.gdg_test_withhold_first_stage
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, ctypes.POINTER(gdg.GdgArgs), ctypes.c_void_p] + \
        [ctypes.c_int] * 5 + [ctypes.c_void_p]
    return f(op_code, ctypes.byref(args), offs.data_ptr(), *dims,
             torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("op", ["fwd", "wgrad"])
def test_withheld_stage_times_out_and_context_survives(cuda_lib, op):
    w = wl.Workload("withhold", E=4, N=512, K=320, ops=(), main_grad_std=1.0)
    h, d = inputs_on(w, DEV, seed=4, sizes=[300, 0, 77, 513], kind=wl.OFFS_ENDS)
    kind = h["kind"]
    assert cuda_lib.gdg_device_error() == 0   # nothing left over from earlier tests
    if op == "fwd":
        args, dims, _, keep = cuda_lib._fwd_args(d["X"], d["W"], d["offs"], None, kind)
        code = cuda_lib.GDG_OP_FWD
    else:
        args, dims, _, keep = cuda_lib._wgrad_args(d["G"], d["X"], d["offs"], None, torch.float32,
                                                   None, False, -1, None, kind)
        code = cuda_lib.GDG_OP_WGRAD
    torch.cuda.synchronize()
    t0 = time.monotonic()
    assert withhold(cuda_lib, code, args, dims, d["offs"]) == 0
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    del keep
    assert cuda_lib.gdg_device_error() == GDG_ETIMEOUT
    assert cuda_lib.gdg_device_error() == 0          # read and cleared
    assert 1.0 < waited < 60.0, waited               # the 2 s in-kernel limit, then a clean exit

    # The context is still usable: the same call without the hook is correct.
    if op == "fwd":
        rows = h["rows"]
        mask = group_rows_mask(h["offs_np"], kind, w.E, rows)
        Y = cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], d["offs"], offs_kind=kind)
        ref = oracle.fwd(h["X"], h["W"], h["offs_np"], kind)
        assert_bf16_close(Y[torch.from_numpy(mask).to(DEV)], ref[mask], "fwd after abort")
    else:
        dW = cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out_dtype=torch.float32,
                                             split_rows=-1, offs_kind=kind)
        ref = oracle.wgrad(h["G"], h["X"], h["offs_np"], w.E, kind)
        assert_fp32_close(dW, ref, "wgrad after abort")
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0
    assert np.isfinite(waited)


def test_error_word_read_on_a_stream_without_host_sync(cuda_lib):
    """gdg_device_error_async copies the word into pinned host memory (and resets it) in stream
    order: after a withheld stage the copy holds GDG_ETIMEOUT, a second read 0; a device-side
    destination works the same way."""
    w = wl.Workload("withhold_async", E=2, N=256, K=256, ops=(), main_grad_std=1.0)
    h, d = inputs_on(w, DEV, seed=6, sizes=[200, 300], kind=wl.OFFS_ENDS)
    assert cuda_lib.gdg_device_error() == 0
    args, dims, _, keep = cuda_lib._fwd_args(d["X"], d["W"], d["offs"], None, wl.OFFS_ENDS)
    stream = torch.cuda.current_stream()
    host = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    dev_word = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    assert withhold(cuda_lib, cuda_lib.GDG_OP_FWD, args, dims, d["offs"]) == 0
    cuda_lib.gdg_device_error_async(host, stream=stream)   # enqueued behind the launch
    stream.synchronize()
    del keep
    assert int(host.item()) == GDG_ETIMEOUT
    cuda_lib.gdg_device_error_async(dev_word, stream=stream)
    assert int(dev_word.item()) == 0                        # the first read reset it
    cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], d["offs"])
    cuda_lib.gdg_device_error_async(host, stream=stream)
    stream.synchronize()
    assert int(host.item()) == 0


def test_error_watch_reports_a_timeout_to_training(cuda_lib):
    """DeviceErrorWatch and the autograd op: a launch whose wait ran out is reported by a later
    forward or backward of grouped_det_mm as GdgError(GDG_ETIMEOUT), with no host sync in the
    op itself; after the report the op runs normally again."""
    w = wl.Workload("withhold_watch", E=2, N=256, K=256, ops=(), main_grad_std=1.0)
    h, d = inputs_on(w, DEV, seed=8, sizes=[150, 350], kind=wl.OFFS_ENDS)
    assert cuda_lib.gdg_device_error() == 0

    # The watch alone: armed behind the timed-out launch, checked once the stream passed it.
    watch = cuda_lib.DeviceErrorWatch(DEV)
    watch.check()                                   # nothing armed: nothing to report
    args, dims, _, keep = cuda_lib._fwd_args(d["X"], d["W"], d["offs"], None, wl.OFFS_ENDS)
    assert withhold(cuda_lib, cuda_lib.GDG_OP_FWD, args, dims, d["offs"]) == 0
    watch.arm()
    torch.cuda.synchronize()
    del keep
    with pytest.raises(cuda_lib.GdgError) as err:
        watch.check()
    assert err.value.status == GDG_ETIMEOUT
    watch.check()                                   # reported once
    assert cuda_lib.gdg_device_error() == 0         # the arm reset the word

    # Through autograd: the backward after the timed-out launch arms the op's watch; the next
    # forward raises.
    x = d["X"].clone().requires_grad_(True)
    wt = d["W"].clone().requires_grad_(True)
    args, dims, _, keep = cuda_lib._fwd_args(d["X"], d["W"], d["offs"], None, wl.OFFS_ENDS)
    assert withhold(cuda_lib, cuda_lib.GDG_OP_FWD, args, dims, d["offs"]) == 0
    y = cuda_lib.grouped_det_mm(x, wt, d["offs"])
    y.backward(d["G"])
    torch.cuda.synchronize()
    del keep
    with pytest.raises(cuda_lib.GdgError) as err:
        cuda_lib.grouped_det_mm(x, wt, d["offs"])
    assert err.value.status == GDG_ETIMEOUT
    # Reported once; the op then matches the oracle again.
    y = cuda_lib.grouped_det_mm(x.detach(), wt.detach(), d["offs"])
    ref = oracle.fwd(h["X"], h["W"], h["offs_np"], wl.OFFS_ENDS)
    assert_bf16_close(y, ref, "fwd after the reported timeout")
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0
