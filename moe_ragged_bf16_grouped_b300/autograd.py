"""Autograd over the C ABI: ``grouped_det_mm(x, w, offs, *, fuse_wgrad_accumulation=False)``.

The computation table of the "Cake ragged BF16 grouped GEMM (experimental)" docs page, wired for
training: the forward is ``grouped_det_gemm_fwd`` (Y[g] = X[g] @ W[e].T), the backward runs
``grouped_det_gemm_dgrad`` for x and ``grouped_det_gemm_wgrad`` for w.  Every step is one of the
library's kernels; this module only routes tensors.

``fuse_wgrad_accumulation=True`` follows the Megatron / Transformer Engine ``main_grad``
convention that the MoE grouped GEMM pull request adopts for the deterministic wrapper
(section "Deterministic weight-gradient accumulation"):

- ``w.main_grad`` (fp32 or bf16, w's shape and device, unit stride along its last dimension; a
  strided view is fine) is checked when the forward runs and read again by the backward;
- the backward adds the deterministic dW into it with the fused accumulate (the bits of
  ``main_grad.add_(dW)``), every time it runs: ``retain_graph`` and a second backward add twice,
  and so does ``torch.autograd.grad`` whose inputs exclude w;
- it then returns a fresh placeholder gradient for w when w has the attribute
  ``grad_added_to_main_grad`` (which it sets to True; zeros when ``w.zero_out_wgrad`` is true,
  else uninitialised), and None otherwise;
- ``create_graph`` (a differentiable backward), ``torch.jit.trace`` and ``torch.compile`` raise
  NotImplementedError;
- a reentrant activation checkpoint (``torch.utils.checkpoint`` with ``use_reentrant=True``)
  raises ValueError when its forward first runs the fused op; non-reentrant and nested
  non-reentrant checkpoints work like any autograd graph (the backward adds once).

Without fusion, w's gradient is dW in w's dtype (bf16), under any checkpoint.

Every backward arms a ``DeviceErrorWatch`` for its device after its launches, and every forward
and backward first checks the watch: a launch whose in-kernel wait ran out (its outputs are
unspecified) raises ``GdgError`` in a later call instead of letting training go on silently,
with no host synchronisation.
"""
from __future__ import annotations

import sys

import torch

_gdg = sys.modules[__package__]


def _check_main_grad(w: torch.Tensor) -> torch.Tensor:
    mg = getattr(w, "main_grad", None)
    if mg is None:
        raise ValueError("fuse_wgrad_accumulation=True needs w.main_grad")
    if mg.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"w.main_grad must be float32 or bfloat16, got {mg.dtype}")
    if tuple(mg.shape) != tuple(w.shape) or mg.device != w.device:
        raise ValueError("w.main_grad must have w's shape and device")
    if mg.stride(-1) != 1:
        raise ValueError("w.main_grad must have unit stride along its last dimension")
    return mg


def _reentrant_checkpoint_code():
    try:
        from torch.utils.checkpoint import CheckpointFunction
    except ImportError:   # a torch without the reentrant checkpoint function
        return ()
    return (CheckpointFunction.forward.__code__, CheckpointFunction.backward.__code__)


def _in_reentrant_checkpoint() -> bool:
    """True when called (at any depth) from the reentrant checkpoint's forward or its
    recomputing backward."""
    codes = _reentrant_checkpoint_code()
    f = sys._getframe(1)
    while f is not None:
        if f.f_code in codes:
            return True
        f = f.f_back
    return False


def _in_checkpoint_recompute() -> bool:
    """True while a non-reentrant checkpoint recomputes its forward inside a backward (its
    saved-tensor unpack hook re-runs the function; the inputs there are recomputed aliases)."""
    f = sys._getframe(1)
    while f is not None:
        c = f.f_code
        if c.co_name in ("recompute_fn", "unpack_hook") and \
                c.co_filename.replace("\\", "/").endswith("torch/utils/checkpoint.py"):
            return True
        f = f.f_back
    return False


_watches = {}


def _watch(device: torch.device):
    """The error watch of this device (one per device, created on first use); None off CUDA
    (the library refuses such tensors itself)."""
    if device.type != "cuda":
        return None
    key = device.index if device.index is not None else torch.cuda.current_device()
    w = _watches.get(key)
    if w is None:
        w = _watches[key] = _gdg.DeviceErrorWatch(torch.device("cuda", key))
    return w


def _refuse_tracing():
    if torch.jit.is_tracing() or torch.compiler.is_compiling():
        raise NotImplementedError("grouped_det_mm cannot be traced or compiled")


class GroupedDetMm(torch.autograd.Function):
    """Y = grouped fwd(x, w, offs); backward: dgrad for x, wgrad (or fused main_grad
    accumulation) for w.  Inputs are bf16 and contiguous; offs is int32 on the same device."""

    @staticmethod
    def forward(ctx, x, w, offs, fuse_wgrad_accumulation=False):
        if not isinstance(fuse_wgrad_accumulation, bool):
            raise ValueError("fuse_wgrad_accumulation must be a bool")
        _refuse_tracing()
        if fuse_wgrad_accumulation:
            if _in_reentrant_checkpoint():
                raise ValueError("fuse_wgrad_accumulation=True cannot run under a reentrant "
                                 "activation checkpoint; use use_reentrant=False")
            # A checkpoint's recomputation only regenerates saved tensors for the node recorded
            # by the first forward (whose weight object the backward uses); its w is an alias
            # without main_grad.
            if not (getattr(w, "main_grad", None) is None and _in_checkpoint_recompute()):
                _check_main_grad(w)
        watch = _watch(x.device)
        if watch is not None:
            watch.check()
        y = _gdg.grouped_det_gemm_fwd(x, w, offs)
        ctx.save_for_backward(x, w, offs)
        ctx.fuse = fuse_wgrad_accumulation
        # The fused backward reads main_grad (and sets grad_added_to_main_grad) on the weight
        # object itself: under a non-reentrant checkpoint the saved w comes back as a
        # recomputed alias without those attributes.  w's own history lies upstream of this
        # node, so holding it here makes no reference cycle.
        ctx.weight = w if fuse_wgrad_accumulation else None
        return y

    @staticmethod
    def backward(ctx, dy):
        if torch.is_grad_enabled():
            raise NotImplementedError("grouped_det_mm does not support create_graph")
        x, w, offs = ctx.saved_tensors
        watch = _watch(x.device)
        if watch is not None:
            watch.check()
        dy = dy.contiguous()
        dx = dw = None
        if ctx.needs_input_grad[0]:
            dx = _gdg.grouped_det_gemm_dgrad(dy, w, offs)
        if ctx.needs_input_grad[1]:
            if ctx.fuse:
                wp = ctx.weight
                mg = _check_main_grad(wp)
                _gdg.grouped_det_gemm_wgrad(dy, x, offs, out=mg, accumulate=True)
                if hasattr(wp, "grad_added_to_main_grad"):
                    wp.grad_added_to_main_grad = True
                    if getattr(wp, "zero_out_wgrad", False):
                        dw = torch.zeros(w.shape, dtype=w.dtype, device=w.device)
                    else:
                        dw = torch.empty(w.shape, dtype=w.dtype, device=w.device)
            else:
                dw = _gdg.grouped_det_gemm_wgrad(dy, x, offs, out_dtype=w.dtype)
        # The forward's launch and this backward's are behind this point on the stream.
        if watch is not None:
            with torch.cuda.device(x.device):
                watch.arm()
        return dx, dw, None, None


def grouped_det_mm(x: torch.Tensor, w: torch.Tensor, offs: torch.Tensor, *,
                   fuse_wgrad_accumulation: bool = False) -> torch.Tensor:
    """Ragged grouped matmul Y[g] = X[g] @ W[e].T with deterministic gradients (offs: int32
    cumulative ends of the groups)."""
    return GroupedDetMm.apply(x, w, offs, fuse_wgrad_accumulation)
