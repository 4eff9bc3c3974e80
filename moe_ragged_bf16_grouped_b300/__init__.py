"""Deterministic ragged BF16 grouped GEMM for B300 -- Python binding of libgdg.so.

The functions below carry the C ABI's names (include/gdg.h) and only marshal
arguments: they read shapes and pointers off torch tensors, allocate missing
outputs or workspace with torch, and pass everything to the CUDA library on
the current stream.  All computation happens in the library's kernels.  There
is no fallback: importing this package fails if libgdg.so is missing.

Operations (computation table of the "Cake ragged BF16 grouped GEMM
(experimental)" docs page; accumulate from the MoE grouped GEMM pull request):

    grouped_det_gemm_fwd(x, w, offs)     Y[g]  = X[g] @ W[e].T   -> [rows, N] bf16
    grouped_det_gemm_dgrad(g, w, offs)   dX[g] = G[g] @ W[e]     -> [rows, K] bf16
    grouped_det_gemm_wgrad(g, x, offs)   dW[e] = G[g].T @ X[g]   -> [E, N, K] bf16/fp32
                                        (accumulate=True: out[e] += G[g].T @ X[g])
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "GDG_OFFS_ENDS", "GDG_OFFS_INDPTR", "GDG_OP_FWD", "GDG_OP_DGRAD", "GDG_OP_WGRAD",
    "GdgError", "grouped_det_gemm_fwd", "grouped_det_gemm_dgrad", "grouped_det_gemm_wgrad",
    "grouped_det_gemm_workspace_bytes", "grouped_det_gemm_auto_split_rows",
    "grouped_det_gemm_wgrad_noalloc", "GDG_NOALLOC_SCRATCH_BYTES", "GroupedDetGemmPlan",
    "prepare_grouped_det_gemm_fwd", "prepare_grouped_det_gemm_dgrad",
    "prepare_grouped_det_gemm_wgrad", "grouped_det_mm", "GroupedDetMm", "DeviceErrorWatch",
    "gdg_status_string", "gdg_device_error", "gdg_device_error_async", "library_path",
    "grouped_gemm_wgrad", "grouped_gemm_wgrad_workspace_bytes",
]

GDG_OK, GDG_EINVAL, GDG_EALIGN, GDG_EOVERLAP, GDG_EWORKSPACE, GDG_ECUDA, GDG_ETIMEOUT = range(7)
GDG_BF16, GDG_FP32 = 0, 1
GDG_OFFS_ENDS, GDG_OFFS_INDPTR = 0, 1
GDG_OP_FWD, GDG_OP_DGRAD, GDG_OP_WGRAD = 0, 1, 2
GDG_NOALLOC_SCRATCH_BYTES = 16 << 20

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgdg.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is not built; run `python -m moe_ragged_bf16_grouped_b300.build`")
_lib = ctypes.CDLL(_LIB_PATH)


class GdgArgs(ctypes.Structure):
    _fields_ = [("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("rows", ctypes.c_int64), ("offs_kind", ctypes.c_int32),
                ("split_rows", ctypes.c_int32), ("out_ld", ctypes.c_int64),
                ("out_es", ctypes.c_int64)]


for _name in ("grouped_det_gemm_fwd", "grouped_det_gemm_dgrad", "grouped_det_gemm_wgrad",
              "grouped_det_gemm_wgrad_noalloc"):
    _f = getattr(_lib, _name)
    _f.restype = ctypes.c_int
    _f.argtypes = [ctypes.POINTER(GdgArgs), ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
_lib.grouped_gemm_wgrad.restype = ctypes.c_int
_lib.grouped_gemm_wgrad.argtypes = [ctypes.POINTER(GdgArgs), ctypes.c_void_p, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_void_p]
_lib.grouped_gemm_wgrad_workspace_bytes.restype = ctypes.c_size_t
_lib.grouped_gemm_wgrad_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int32]
_lib.grouped_det_gemm_workspace_bytes.restype = ctypes.c_size_t
_lib.grouped_det_gemm_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_int32]
_lib.grouped_det_gemm_auto_split_rows.restype = ctypes.c_int32
_lib.grouped_det_gemm_auto_split_rows.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int]
_lib.gdg_status_string.restype = ctypes.c_char_p
_lib.gdg_status_string.argtypes = [ctypes.c_int]
_lib.gdg_device_error.restype = ctypes.c_int
_lib.gdg_device_error.argtypes = []
_lib.gdg_device_error_async.restype = ctypes.c_int
_lib.gdg_device_error_async.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
_lib.gdg_plan_create.restype = ctypes.c_int
_lib.gdg_plan_create.argtypes = [ctypes.c_int, ctypes.POINTER(GdgArgs), ctypes.c_void_p,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)]
_lib.gdg_plan_launch.restype = ctypes.c_int
_lib.gdg_plan_launch.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
_lib.gdg_plan_destroy.restype = None
_lib.gdg_plan_destroy.argtypes = [ctypes.c_void_p]


def library_path() -> str:
    return _LIB_PATH


class GdgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {gdg_status_string(status)} (status {status})")


def gdg_status_string(status: int) -> str:
    return _lib.gdg_status_string(status).decode()


def gdg_device_error() -> int:
    """Synchronises the device and returns (and clears) the device error word."""
    return _lib.gdg_device_error()


def gdg_device_error_async(dst: torch.Tensor, stream=None) -> torch.Tensor:
    """Enqueues on ``stream`` a copy of the device error word into ``dst`` (one int32 element,
    on the device or in pinned host memory) and a reset of the word, with no host
    synchronisation.  Once the stream has passed that point ``dst`` holds 0 (GDG_OK) or 6
    (GDG_ETIMEOUT: a launch stopped early and its outputs are unspecified)."""
    if not isinstance(dst, torch.Tensor) or dst.dtype != torch.int32 or dst.numel() < 1:
        raise ValueError("dst must be an int32 tensor with at least one element")
    if not dst.is_cuda and not dst.is_pinned():
        raise ValueError("dst must be on the device or in pinned host memory")
    device = dst.device if dst.is_cuda else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(device):
        st = _lib.gdg_device_error_async(dst.data_ptr(), _stream_ptr(stream, device))
    if st != GDG_OK:
        raise GdgError(st, "gdg_device_error_async")
    return dst


class DeviceErrorWatch:
    """A check of one device's error word that never blocks the host.

    ``arm(stream)`` enqueues on the stream a copy of the word into a slot of pinned host memory,
    and its reset (``gdg_device_error_async``), and records an event behind them.  ``check()``
    reads every armed slot whose event has completed, skipping the others, and raises
    ``GdgError`` (``GDG_ETIMEOUT``: a launch stopped early and left its outputs unspecified) if
    one of them held a set word.  A timed-out launch is therefore reported by the first
    ``check()`` after the stream has passed the next ``arm()``, without any synchronisation.
    Neither call does anything while the current stream is being captured into a graph."""

    def __init__(self, device, slots: int = 8):
        self.device = torch.device(device)
        if self.device.type != "cuda":
            raise ValueError("DeviceErrorWatch needs a CUDA device")
        self._words = torch.zeros(slots, dtype=torch.int32).pin_memory()
        self._events = [None] * slots
        self._next = 0

    def _read(self, i: int) -> None:
        self._events[i] = None
        word = int(self._words[i])
        if word != GDG_OK:
            self._words[i] = GDG_OK
            raise GdgError(word, "device error word (DeviceErrorWatch)")

    def check(self) -> None:
        if torch.cuda.is_current_stream_capturing():
            return
        for i, ev in enumerate(self._events):
            if ev is not None and ev.query():
                self._read(i)

    def arm(self, stream=None) -> None:
        if torch.cuda.is_current_stream_capturing():
            return
        i = self._next
        if self._events[i] is not None:      # every slot in flight: the oldest must land first
            self._events[i].synchronize()
            self._read(i)
        self._next = (i + 1) % len(self._events)
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        gdg_device_error_async(self._words[i:i + 1], stream)
        ev = torch.cuda.Event()
        ev.record(stream)
        self._events[i] = ev


def grouped_det_gemm_workspace_bytes(op: int, rows: int, E: int, N: int, K: int,
                                     out_dtype: torch.dtype = torch.bfloat16,
                                     accumulate: bool = False, split_rows: int = 0) -> int:
    n = _lib.grouped_det_gemm_workspace_bytes(op, rows, E, N, K, _dtype_code(out_dtype),
                                              int(accumulate), split_rows)
    if n == ctypes.c_size_t(-1).value:
        raise GdgError(GDG_EINVAL, "grouped_det_gemm_workspace_bytes")
    return n


def grouped_det_gemm_auto_split_rows(rows: int, E: int, N: int, K: int) -> int:
    return _lib.grouped_det_gemm_auto_split_rows(rows, E, N, K)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return GDG_BF16
    if dt == torch.float32:
        return GDG_FP32
    raise ValueError(f"unsupported output dtype {dt}")


def _check_operand(t: torch.Tensor, name: str, dtype=torch.bfloat16, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_out(t: torch.Tensor, dtype, ndim: int):
    """An output may be a strided view (unit stride along its last dimension); the library
    checks alignment and that no two elements share memory."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("out must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"out must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"out must have {ndim} dimensions, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError("out must be on a CUDA device")
    if t.numel() and t.stride(-1) != 1:
        raise ValueError("out must have unit stride along its last dimension")


def _out_strides(out: torch.Tensor):
    """(row stride, expert stride) in elements for the C ABI; 0 (dense) where a dimension has
    a single entry, whose stride torch does not pin down."""
    ld = out.stride(-2) if out.shape[-2] > 1 else 0
    es = (out.stride(0) if out.shape[0] > 1 else 0) if out.dim() == 3 else 0
    return ld, es


def _same_device(*tensors):
    dev = tensors[0].device
    for t in tensors[1:]:
        if t is not None and t.device != dev:
            raise ValueError(f"all tensors must be on one device ({dev}, got {t.device})")


def _offs_kind(offs_kind) -> int:
    if offs_kind in (GDG_OFFS_ENDS, "ends", "offs"):
        return GDG_OFFS_ENDS
    if offs_kind in (GDG_OFFS_INDPTR, "indptr", "m_indptr"):
        return GDG_OFFS_INDPTR
    raise ValueError(f"unknown offs_kind {offs_kind!r}")


def _num_groups(offs: torch.Tensor, kind: int) -> int:
    _check_operand(offs, "offs", torch.int32, 1)
    return offs.numel() - (1 if kind == GDG_OFFS_INDPTR else 0)


def _stream_ptr(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _call(fn, name, args, offs, E, N, K, dtype_code, accumulate, stream):
    # The library works on the calling thread's current device: make it the tensors' device.
    with torch.cuda.device(offs.device):
        st = fn(ctypes.byref(args), offs.data_ptr(), E, N, K, dtype_code, int(accumulate), stream)
    if st != GDG_OK:
        raise GdgError(st, name)


def _fwd_args(x, w, offs, out, offs_kind):
    kind = _offs_kind(offs_kind)
    _check_operand(x, "x", ndim=2)
    _check_operand(w, "w", ndim=3)
    E, N, K = w.shape
    if x.shape[1] != K or _num_groups(offs, kind) != E:
        raise ValueError("shape mismatch between x, w and offs")
    if out is None:
        out = torch.empty((x.shape[0], N), dtype=torch.bfloat16, device=x.device)
    _check_out(out, torch.bfloat16, 2)
    if tuple(out.shape) != (x.shape[0], N):
        raise ValueError("out must be [rows, N]")
    _same_device(offs, x, w, out)
    args = GdgArgs(x.data_ptr(), w.data_ptr(), out.data_ptr(), None, 0, x.shape[0], kind, 0,
                   *_out_strides(out))
    return args, (E, N, K, GDG_BF16, 0), out, (x, w, offs, out)


def _dgrad_args(g, w, offs, out, offs_kind):
    kind = _offs_kind(offs_kind)
    _check_operand(g, "g", ndim=2)
    _check_operand(w, "w", ndim=3)
    E, N, K = w.shape
    if g.shape[1] != N or _num_groups(offs, kind) != E:
        raise ValueError("shape mismatch between g, w and offs")
    if out is None:
        out = torch.empty((g.shape[0], K), dtype=torch.bfloat16, device=g.device)
    _check_out(out, torch.bfloat16, 2)
    if tuple(out.shape) != (g.shape[0], K):
        raise ValueError("out must be [rows, K]")
    _same_device(offs, g, w, out)
    args = GdgArgs(g.data_ptr(), w.data_ptr(), out.data_ptr(), None, 0, g.shape[0], kind, 0,
                   *_out_strides(out))
    return args, (E, N, K, GDG_BF16, 0), out, (g, w, offs, out)


def _wgrad_args(g, x, offs, out, out_dtype, num_groups, accumulate, split_rows, workspace,
                offs_kind):
    kind = _offs_kind(offs_kind)
    _check_operand(g, "g", ndim=2)
    _check_operand(x, "x", ndim=2)
    rows, N = g.shape
    if x.shape[0] != rows:
        raise ValueError("g and x must have the same number of rows")
    K = x.shape[1]
    E = _num_groups(offs, kind)
    if num_groups is not None and num_groups != E:
        raise ValueError("num_groups does not match offs")
    if out is None:
        if accumulate:
            raise ValueError("accumulate=True needs out")
        out = torch.empty((E, N, K), dtype=out_dtype or torch.bfloat16, device=g.device)
    if out_dtype is not None and out_dtype != out.dtype:
        raise ValueError("out_dtype must be None or out.dtype")
    _check_out(out, out.dtype, 3)
    if tuple(out.shape) != (E, N, K):
        raise ValueError("out must be [E, N, K]")
    code = _dtype_code(out.dtype)
    _same_device(offs, g, x, out, workspace)
    need = grouped_det_gemm_workspace_bytes(GDG_OP_WGRAD, rows, E, N, K, out.dtype, accumulate,
                                            split_rows)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=g.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = GdgArgs(g.data_ptr(), x.data_ptr(), out.data_ptr(), ws_ptr, ws_bytes, rows, kind,
                   split_rows, *_out_strides(out))
    return args, (E, N, K, code, int(accumulate)), out, (g, x, offs, out, workspace)


def grouped_det_gemm_fwd(x: torch.Tensor, w: torch.Tensor, offs: torch.Tensor,
                         out: torch.Tensor | None = None, *, offs_kind=GDG_OFFS_ENDS,
                         stream=None) -> torch.Tensor:
    """Y[rows, N] with Y[g] = X[g] @ W[e].T for every group (rows outside all groups
    are left as they are in ``out``)."""
    args, dims, out, _ = _fwd_args(x, w, offs, out, offs_kind)
    _call(_lib.grouped_det_gemm_fwd, "grouped_det_gemm_fwd", args, offs, *dims,
          _stream_ptr(stream, x.device))
    return out


def grouped_det_gemm_dgrad(g: torch.Tensor, w: torch.Tensor, offs: torch.Tensor,
                           out: torch.Tensor | None = None, *, offs_kind=GDG_OFFS_ENDS,
                           stream=None) -> torch.Tensor:
    """dX[rows, K] with dX[g] = G[g] @ W[e] (W as stored)."""
    args, dims, out, _ = _dgrad_args(g, w, offs, out, offs_kind)
    _call(_lib.grouped_det_gemm_dgrad, "grouped_det_gemm_dgrad", args, offs, *dims,
          _stream_ptr(stream, g.device))
    return out


def grouped_det_gemm_wgrad(g: torch.Tensor, x: torch.Tensor, offs: torch.Tensor,
                           out: torch.Tensor | None = None, out_dtype: torch.dtype | None = None,
                           num_groups: int | None = None, *, accumulate: bool = False,
                           split_rows: int = 0, workspace: torch.Tensor | None = None,
                           offs_kind=GDG_OFFS_ENDS, stream=None) -> torch.Tensor:
    """dW[E, N, K] with dW[e] = G[g].T @ X[g]; with ``accumulate`` the result is added
    into ``out`` (bitwise ``out.add_(dW)`` in out's dtype)."""
    args, dims, out, _ = _wgrad_args(g, x, offs, out, out_dtype, num_groups, accumulate,
                                     split_rows, workspace, offs_kind)
    _call(_lib.grouped_det_gemm_wgrad, "grouped_det_gemm_wgrad", args, offs, *dims,
          _stream_ptr(stream, g.device))
    return out


class GroupedDetGemmPlan:
    """A prepared launch (``gdg_plan_create``): the call's checks ran and its buffers, kernel
    form and grid are bound.  ``launch()`` enqueues the call's kernels on a stream with no
    other host work; it allocates nothing, never synchronises and can be captured in a CUDA
    graph.  New values written into the bound tensors (offsets included) are honoured by every
    later launch or replay; with accumulate each launch adds again.  The plan keeps its tensors
    alive.  ``out`` is the bound output tensor."""

    def __init__(self, op: int, args: GdgArgs, dims, offs: torch.Tensor, out: torch.Tensor,
                 keep, name: str):
        self.out = out
        self._keep = keep
        self._device = out.device
        h = ctypes.c_void_p()
        with torch.cuda.device(self._device):
            st = _lib.gdg_plan_create(op, ctypes.byref(args), offs.data_ptr(), *dims,
                                      ctypes.byref(h))
        if st != GDG_OK:
            raise GdgError(st, name)
        self._h = h

    def launch(self, stream=None) -> torch.Tensor:
        with torch.cuda.device(self._device):
            st = _lib.gdg_plan_launch(self._h, _stream_ptr(stream, self._device))
        if st != GDG_OK:
            raise GdgError(st, "gdg_plan_launch")
        return self.out

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            _lib.gdg_plan_destroy(h)
            self._h = None


def prepare_grouped_det_gemm_fwd(x, w, offs, out=None, *, offs_kind=GDG_OFFS_ENDS):
    """Prepared form of grouped_det_gemm_fwd (same arguments)."""
    args, dims, out, keep = _fwd_args(x, w, offs, out, offs_kind)
    return GroupedDetGemmPlan(GDG_OP_FWD, args, dims, offs, out, keep, "prepare_grouped_det_gemm_fwd")


def prepare_grouped_det_gemm_dgrad(g, w, offs, out=None, *, offs_kind=GDG_OFFS_ENDS):
    """Prepared form of grouped_det_gemm_dgrad (same arguments)."""
    args, dims, out, keep = _dgrad_args(g, w, offs, out, offs_kind)
    return GroupedDetGemmPlan(GDG_OP_DGRAD, args, dims, offs, out, keep,
                              "prepare_grouped_det_gemm_dgrad")


def prepare_grouped_det_gemm_wgrad(g, x, offs, out=None, out_dtype=None, num_groups=None, *,
                                   accumulate=False, split_rows=0, workspace=None,
                                   offs_kind=GDG_OFFS_ENDS):
    """Prepared form of grouped_det_gemm_wgrad (same arguments); the split form's workspace
    is allocated here when not given and bound to the plan."""
    args, dims, out, keep = _wgrad_args(g, x, offs, out, out_dtype, num_groups, accumulate,
                                        split_rows, workspace, offs_kind)
    return GroupedDetGemmPlan(GDG_OP_WGRAD, args, dims, offs, out, keep,
                              "prepare_grouped_det_gemm_wgrad")


def grouped_det_gemm_wgrad_noalloc(g: torch.Tensor, x: torch.Tensor, offs: torch.Tensor,
                                   out: torch.Tensor, *, accumulate: bool = False,
                                   split_rows: int = 0, offs_kind=GDG_OFFS_ENDS,
                                   stream=None) -> torch.Tensor:
    """Split-form weight gradient into ``out`` using only the library's fixed device
    scratch (GDG_NOALLOC_SCRATCH_BYTES) instead of a caller workspace: for callers that
    must not allocate device memory while computing it.  ``out`` is required; nothing is
    allocated here either.  Calls that overlap on the GPU share the scratch and race."""
    kind = _offs_kind(offs_kind)
    _check_operand(g, "g", ndim=2)
    _check_operand(x, "x", ndim=2)
    rows, N = g.shape
    if x.shape[0] != rows:
        raise ValueError("g and x must have the same number of rows")
    K = x.shape[1]
    E = _num_groups(offs, kind)
    _check_out(out, out.dtype, 3)
    if tuple(out.shape) != (E, N, K):
        raise ValueError("out must be [E, N, K]")
    _same_device(offs, g, x, out)
    args = GdgArgs(g.data_ptr(), x.data_ptr(), out.data_ptr(), None, 0, rows, kind, split_rows,
                   *_out_strides(out))
    _call(_lib.grouped_det_gemm_wgrad_noalloc, "grouped_det_gemm_wgrad_noalloc", args, offs, E,
          N, K, _dtype_code(out.dtype), int(accumulate), _stream_ptr(stream, g.device))
    return out


def grouped_gemm_wgrad_workspace_bytes(rows: int, E: int, N: int, K: int,
                                       out_dtype: torch.dtype = torch.bfloat16,
                                       accumulate: bool = False, split_rows: int = 0) -> int:
    n = _lib.grouped_gemm_wgrad_workspace_bytes(rows, E, N, K, _dtype_code(out_dtype),
                                                int(accumulate), split_rows)
    if n == ctypes.c_size_t(-1).value:
        raise GdgError(GDG_EINVAL, "grouped_gemm_wgrad_workspace_bytes")
    return n


def grouped_gemm_wgrad(g: torch.Tensor, x: torch.Tensor, offs: torch.Tensor,
                       out: torch.Tensor | None = None, out_dtype: torch.dtype | None = None,
                       num_groups: int | None = None, *, deterministic=True,
                       accumulate: bool = False, split_rows: int = 0,
                       workspace: torch.Tensor | None = None, offs_kind=GDG_OFFS_ENDS,
                       stream=None) -> torch.Tensor:
    """Non-deterministic weight gradient (the MoE grouped GEMM pull request's non-deterministic
    package, "Mode rules"): as grouped_det_gemm_wgrad, except that the row chunks of the split
    form are added with unordered fp32 atomics, so dW varies in its low bits from run to run.

    ``deterministic`` is keyword-only and only the bool False runs; any other value raises
    ValueError naming the deterministic entry.  Under ``torch.use_deterministic_algorithms(True)``
    a call that takes the split form raises RuntimeError before launching (``warn_only=True``:
    one UserWarning, then the launch); the unsplit form runs in a fixed order and never alerts."""
    if deterministic is not False:
        raise ValueError("grouped_gemm_wgrad is the non-deterministic entry: pass "
                         "deterministic=False for the non-deterministic path, or call "
                         "grouped_det_gemm_wgrad for the deterministic one")
    kind = _offs_kind(offs_kind)
    _check_operand(g, "g", ndim=2)
    _check_operand(x, "x", ndim=2)
    rows, N = g.shape
    if x.shape[0] != rows:
        raise ValueError("g and x must have the same number of rows")
    K = x.shape[1]
    E = _num_groups(offs, kind)
    if num_groups is not None and num_groups != E:
        raise ValueError("num_groups does not match offs")
    if out is None:
        if accumulate:
            raise ValueError("accumulate=True needs out")
        out = torch.empty((E, N, K), dtype=out_dtype or torch.bfloat16, device=g.device)
    if out_dtype is not None and out_dtype != out.dtype:
        raise ValueError("out_dtype must be None or out.dtype")
    _check_out(out, out.dtype, 3)
    if tuple(out.shape) != (E, N, K):
        raise ValueError("out must be [E, N, K]")
    _same_device(offs, g, x, out, workspace)
    resolved = split_rows if split_rows != 0 else grouped_det_gemm_auto_split_rows(rows, E, N, K)
    if resolved > 0 and rows > 0 and torch.are_deterministic_algorithms_enabled():
        msg = ("grouped_gemm_wgrad adds the row chunks of its split form in an unordered way; "
               "grouped_det_gemm_wgrad is the deterministic entry")
        if torch.is_deterministic_algorithms_warn_only_enabled():
            import warnings
            warnings.warn(msg, UserWarning, stacklevel=2)
        else:
            raise RuntimeError(msg)
    need = grouped_gemm_wgrad_workspace_bytes(rows, E, N, K, out.dtype, accumulate, split_rows)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=g.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = GdgArgs(g.data_ptr(), x.data_ptr(), out.data_ptr(), ws_ptr, ws_bytes, rows, kind,
                   split_rows, *_out_strides(out))
    with torch.cuda.device(offs.device):
        st = _lib.grouped_gemm_wgrad(ctypes.byref(args), offs.data_ptr(), E, N, K,
                                     _dtype_code(out.dtype), int(accumulate), 0,
                                     _stream_ptr(stream, g.device))
    if st != GDG_OK:
        raise GdgError(st, "grouped_gemm_wgrad")
    return out


from .autograd import GroupedDetMm, grouped_det_mm  # noqa: E402  (needs the functions above)
