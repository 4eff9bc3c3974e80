"""C ABI checks that need no GPU: the library loads, exports every function that
include/gdg.h declares, and refuses bad arguments on the host before any CUDA
call (the checks of the accumulate section of the MoE grouped GEMM pull request
run "before anything is allocated or bound")."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdg.h")
LIB = os.path.join(ROOT, "moe_ragged_bf16_grouped_b300", "libgdg.so")


@pytest.fixture(scope="module")
def lib():
    return ctypes.CDLL(LIB)


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"GDG_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    assert {"grouped_det_gemm_fwd", "grouped_det_gemm_dgrad", "grouped_det_gemm_wgrad",
            "grouped_det_gemm_workspace_bytes", "gdg_status_string"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


class Args(ctypes.Structure):
    _fields_ = [("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("rows", ctypes.c_int64), ("offs_kind", ctypes.c_int32),
                ("split_rows", ctypes.c_int32),
                ("out_ld", ctypes.c_int64), ("out_es", ctypes.c_int64)]


def call(lib, op, args, offs, E, N, K, dtype=0, acc=0):
    f = getattr(lib, op)
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(Args), ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    return f(ctypes.byref(args) if args is not None else None, offs, E, N, K, dtype, acc, None)


EINVAL, EALIGN, EOVERLAP, EWORKSPACE = 1, 2, 3, 4
# Fake, 16-byte aligned device addresses: the host checks never dereference them.
A, B, OUT, OFFS = 0x100000, 0x40000000, 0x80000000, 0xC0000000


def good(rows=512, kind=0, split=0):
    return Args(A, B, OUT, None, 0, rows, kind, split)


@pytest.mark.parametrize("op", ["grouped_det_gemm_fwd", "grouped_det_gemm_dgrad",
                                "grouped_det_gemm_wgrad"])
def test_refusals_before_launch(lib, op):
    assert call(lib, op, None, OFFS, 4, 256, 256) == EINVAL
    assert call(lib, op, good(), None, 4, 256, 256) == EINVAL
    assert call(lib, op, good(), OFFS, 0, 256, 256) == EINVAL
    assert call(lib, op, good(), OFFS, 1025, 256, 256) == EINVAL
    assert call(lib, op, good(rows=-1), OFFS, 4, 256, 256) == EINVAL
    assert call(lib, op, good(kind=2), OFFS, 4, 256, 256) == EINVAL
    assert call(lib, op, good(), OFFS, 4, 132, 256) == EALIGN      # N % 8: rows not 16-byte aligned
    assert call(lib, op, good(), OFFS, 4, 256, 100) == EALIGN      # K % 8
    assert call(lib, op, good(), OFFS, 4, 256, 256, dtype=7) == EINVAL
    bad = good()
    bad.out = OUT + 8
    assert call(lib, op, bad, OFFS, 4, 256, 256) == EALIGN
    ovl = good()
    ovl.out = A + 4096                                             # inside the first operand
    assert call(lib, op, ovl, OFFS, 4, 256, 256) == EOVERLAP


def test_fwd_dgrad_refuse_fp32_and_accumulate(lib):
    for op in ("grouped_det_gemm_fwd", "grouped_det_gemm_dgrad"):
        assert call(lib, op, good(), OFFS, 4, 256, 256, dtype=1) == EINVAL
        assert call(lib, op, good(), OFFS, 4, 256, 256, acc=1) == EINVAL
        assert call(lib, op, good(split=64), OFFS, 4, 256, 256) == EINVAL


def test_wgrad_refusals(lib):
    op = "grouped_det_gemm_wgrad"
    assert call(lib, op, good(split=100), OFFS, 4, 256, 256) == EINVAL      # not a multiple of 64
    assert call(lib, op, good(split=-2), OFFS, 4, 256, 256) == EINVAL
    assert call(lib, op, good(), OFFS, 4, 256, 256, acc=2) == EINVAL
    assert call(lib, op, good(split=64), OFFS, 4, 256, 256) == EWORKSPACE   # split needs scratch
    ovl = good()
    ovl.out = OFFS - 64                                                     # dW covers the offsets
    assert call(lib, op, ovl, OFFS, 4, 256, 256) == EOVERLAP
    ws = good(split=64)
    ws.workspace, ws.workspace_bytes = A + 4096, 1 << 30                    # scratch over an input
    assert call(lib, op, ws, OFFS, 4, 256, 256) == EOVERLAP


def strided(ld=0, es=0, rows=512):
    a = good(rows=rows)
    a.out_ld, a.out_es = ld, es
    return a


@pytest.mark.parametrize("op", ["grouped_det_gemm_fwd", "grouped_det_gemm_dgrad"])
def test_output_stride_refusals_fwd_dgrad(lib, op):
    """Row strides of Y / dX: 16-byte multiples that reach past a row; no expert stride."""
    assert call(lib, op, strided(ld=-8), OFFS, 4, 256, 256) == EINVAL
    assert call(lib, op, strided(es=8), OFFS, 4, 256, 256) == EINVAL         # fwd/dgrad: 2-D out
    assert call(lib, op, strided(ld=260), OFFS, 4, 256, 256) == EALIGN       # 520 B rows
    assert call(lib, op, strided(ld=248), OFFS, 4, 256, 256) == EOVERLAP     # rows overlap


def test_output_stride_refusals_wgrad(lib):
    """dW / main_grad strides: aligned, and no two of the E x N x K elements at one address."""
    op = "grouped_det_gemm_wgrad"
    assert call(lib, op, strided(ld=-8), OFFS, 4, 256, 256) == EINVAL
    assert call(lib, op, strided(ld=260), OFFS, 4, 256, 256) == EALIGN       # bf16: 520 B
    assert call(lib, op, strided(ld=258), OFFS, 4, 256, 256, dtype=1) == EALIGN   # fp32: 1032 B
    assert call(lib, op, strided(ld=128), OFFS, 4, 256, 256) == EOVERLAP     # rows overlap
    # experts 8 elements short of N rows: the last row of expert e meets expert e + 1
    assert call(lib, op, strided(ld=256, es=256 * 256 - 8), OFFS, 4, 256, 256) == EOVERLAP
    # experts interleaved row by row but rows only 2 experts apart: rows collide
    assert call(lib, op, strided(ld=512, es=256), OFFS, 4, 256, 256) == EOVERLAP
    # the same refusals hold for accumulate (main_grad views) and through the plan API
    assert call(lib, op, strided(ld=128), OFFS, 4, 256, 256, dtype=1, acc=1) == EOVERLAP


def test_workspace_bytes_and_auto_form(lib):
    f = lib.grouped_det_gemm_workspace_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int32]
    g = lib.grouped_det_gemm_auto_split_rows
    g.restype = ctypes.c_int32
    g.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    assert f(0, 512, 4, 256, 256, 0, 0, 0) == 0 and f(1, 512, 4, 256, 256, 0, 0, 0) == 0
    assert f(2, 512, 4, 256, 256, 1, 0, -1) == 0
    # split rows 64 on [E=4, N=256, K=256]: (N/256)*(K/256) = 1 tile per expert,
    # at most ceil(512/64) + 4 = 12 chunks -> 12 partial tiles of 256 x 256 fp32
    assert f(2, 512, 4, 256, 256, 1, 1, 64) == 12 * 256 * 256 * 4
    assert f(2, 512, 4, 256, 256, 0, 0, 100) == ctypes.c_size_t(-1).value
    assert f(3, 512, 4, 256, 256, 0, 0, 0) == ctypes.c_size_t(-1).value
    # N, K that are not tile multiples round the tiles up: N=264, K=328 -> 2 x 2 tiles per expert
    assert f(2, 512, 4, 264, 328, 1, 1, 64) == 4 * 12 * 256 * 256 * 4
    assert f(2, 512, 4, 260, 328, 1, 1, 64) == ctypes.c_size_t(-1).value   # N % 8
    # the automatic form depends on shapes only
    assert g(16384, 8, 14336, 4096) == -1          # many tiles: unsplit
    assert g(65536, 64, 1536, 2048) == -1
    assert g(512, 4, 256, 256) == -1              # few tiles but short groups: unsplit
    r = g(65536, 4, 256, 256)                      # few tiles, long groups: split
    assert r > 0 and r % 64 == 0
    assert f(2, 65536, 4, 256, 256, 0, 0, 0) == f(2, 65536, 4, 256, 256, 0, 0, r) > 0


def test_status_strings(lib):
    lib.gdg_status_string.restype = ctypes.c_char_p
    for s in range(7):
        assert lib.gdg_status_string(s)
    assert b"unknown" in lib.gdg_status_string(99)


def test_plan_refusals_leave_no_plan(lib):
    """gdg_plan_create runs the entry points' checks on the host and binds nothing on failure."""
    lib.gdg_plan_create.restype = ctypes.c_int
    lib.gdg_plan_create.argtypes = [ctypes.c_int, ctypes.POINTER(Args), ctypes.c_void_p,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)]
    lib.gdg_plan_launch.restype = ctypes.c_int
    lib.gdg_plan_launch.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.gdg_plan_destroy.restype = None
    lib.gdg_plan_destroy.argtypes = [ctypes.c_void_p]
    h = ctypes.c_void_p(1)
    # (op, E, out dtype, accumulate): fp32 fwd, accumulating dgrad, accumulate=2, unknown op,
    # no groups
    for op, E, dtype, acc in ((0, 4, 1, 0), (1, 4, 0, 1), (2, 4, 0, 2), (3, 4, 0, 0), (0, 0, 0, 0)):
        assert lib.gdg_plan_create(op, ctypes.byref(good()), OFFS, E, 256, 256, dtype, acc,
                                   ctypes.byref(h)) == EINVAL
        assert h.value is None
    assert lib.gdg_plan_create(0, ctypes.byref(good()), OFFS, 4, 132, 256, 0, 0,
                               ctypes.byref(h)) == EALIGN
    assert lib.gdg_plan_create(2, ctypes.byref(good(split=64)), OFFS, 4, 256, 256, 0, 0,
                               ctypes.byref(h)) == EWORKSPACE
    assert h.value is None
    assert lib.gdg_plan_create(0, ctypes.byref(good()), OFFS, 4, 256, 256, 0, 0, None) == EINVAL
    assert lib.gdg_plan_launch(None, None) == EINVAL
    lib.gdg_plan_destroy(None)


def test_async_error_read_refuses_null_destination(lib):
    f = lib.gdg_device_error_async
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert f(None, None) == EINVAL          # refused before any CUDA call


def test_error_watch_needs_a_cuda_device():
    """DeviceErrorWatch reads the device error word of a CUDA device only."""
    import moe_ragged_bf16_grouped_b300 as gdg
    with pytest.raises(ValueError):
        gdg.DeviceErrorWatch("cpu")
