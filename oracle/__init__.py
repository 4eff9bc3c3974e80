"""fp64 CPU oracle of the ragged BF16 grouped GEMM -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never does.

Every function restates one row of the computation table on the "Cake ragged
BF16 grouped GEMM (experimental)" docs page (fwd ``Y = X @ W[e].T``, dgrad
``dX = G @ W[e]`` with W as stored, wgrad ``dW[e] = G.T @ X``) with the group
row ranges of that page's intro paragraph, in plain fp64 loops (C, OpenMP over
independent outputs, every sum in ascending index order).  The accumulate mode
follows the deterministic weight-gradient accumulation section of the MoE
grouped GEMM pull request: ``out[e] += G[e].T @ X[e]``.

Pins (tests/test_oracle.py): identity and permutation weights, a dense
block-diagonal numpy matmul on tiny inputs, integer-exact cases, exact zeros
for empty groups, the fwd/dgrad/wgrad adjoint identity, group-splitting
additivity, offsets-convention equivalence and a hand-worked fixture.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

OFFS_ENDS = 0
OFFS_INDPTR = 1

_lib = None
_i64p = ctypes.POINTER(ctypes.c_int64)


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(_build.build())
        u16p = ctypes.c_void_p
        for name in ("gdg_oracle_fwd", "gdg_oracle_dgrad", "gdg_oracle_wgrad"):
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = [u16p, u16p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        for name in ("gdg_oracle_fwd_rows", "gdg_oracle_dgrad_rows"):
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = [u16p, u16p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                          ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
        f = lib.gdg_oracle_wgrad_entries
        f.restype = ctypes.c_int
        f.argtypes = [u16p, u16p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                      ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                      ctypes.c_void_p]
        f = lib.gdg_oracle_wgrad_rows
        f.restype = ctypes.c_int
        f.argtypes = [u16p, u16p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                      ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                      ctypes.c_void_p]
        lib.gdg_oracle_bounds.restype = ctypes.c_int
        lib.gdg_oracle_bounds.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
        lib.gdg_oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


class OracleError(ValueError):
    pass


def _bits(a) -> np.ndarray:
    """bf16 operand as contiguous uint16 bit patterns (torch bf16 tensor or uint16 array)."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        a = a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle operands are bf16 bit patterns (uint16)")
    return a


def _offs(offs) -> np.ndarray:
    if hasattr(offs, "cpu"):
        offs = offs.cpu().numpy()
    return np.ascontiguousarray(offs, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().gdg_oracle_num_threads()


def bounds(offs, kind: int, E: int, rows: int):
    """Row range [start[e], end[e]) of every group (docs page intro paragraph)."""
    o = _offs(offs)
    st = np.zeros(E, np.int64)
    en = np.zeros(E, np.int64)
    if _load().gdg_oracle_bounds(_ptr(o), kind, E, rows, _ptr(st), _ptr(en)):
        raise OracleError("invalid offsets")
    return st, en


def _check(rc):
    if rc == -1:
        raise OracleError("invalid offsets")
    if rc != 0:
        raise MemoryError("oracle allocation failed")


def fwd(X, W, offs, kind: int = OFFS_ENDS, out=None) -> np.ndarray:
    """Y[rows, N] in fp64; rows outside every group keep ``out``'s value (NaN by default)."""
    x, w, o = _bits(X), _bits(W), _offs(offs)
    rows, K = x.shape
    E, N, K2 = w.shape
    assert K2 == K
    Y = np.full((rows, N), np.nan) if out is None else out
    _check(_load().gdg_oracle_fwd(_ptr(x), _ptr(w), _ptr(o), kind, rows, E, N, K, _ptr(Y)))
    return Y


def dgrad(G, W, offs, kind: int = OFFS_ENDS, out=None) -> np.ndarray:
    """dX[rows, K] in fp64; rows outside every group keep ``out``'s value."""
    g, w, o = _bits(G), _bits(W), _offs(offs)
    rows, N = g.shape
    E, N2, K = w.shape
    assert N2 == N
    dX = np.full((rows, K), np.nan) if out is None else out
    _check(_load().gdg_oracle_dgrad(_ptr(g), _ptr(w), _ptr(o), kind, rows, E, N, K, _ptr(dX)))
    return dX


def wgrad(G, X, offs, E: int, kind: int = OFFS_ENDS) -> np.ndarray:
    """dW[E, N, K] in fp64 (exactly zero for an empty group)."""
    g, x, o = _bits(G), _bits(X), _offs(offs)
    rows, N = g.shape
    rows2, K = x.shape
    assert rows2 == rows
    dW = np.empty((E, N, K))
    _check(_load().gdg_oracle_wgrad(_ptr(g), _ptr(x), _ptr(o), kind, rows, E, N, K, _ptr(dW)))
    return dW


def wgrad_accumulate(main_grad, G, X, offs, E: int, kind: int = OFFS_ENDS) -> np.ndarray:
    """``main_grad + dW`` in fp64: the accumulate mode's exact value,
    ``out[e] += G[e].T @ X[e]`` (MoE grouped GEMM pull request, deterministic
    weight-gradient accumulation)."""
    mg = np.asarray(main_grad.detach().cpu().numpy() if hasattr(main_grad, "detach") else main_grad,
                    dtype=np.float64)
    return mg + wgrad(G, X, offs, E, kind)


def fwd_rows(X, W, offs, row_ids, kind: int = OFFS_ENDS):
    """Y for the listed rows only: (Y[len(row_ids), N], group of each row or -1)."""
    x, w, o = _bits(X), _bits(W), _offs(offs)
    ids = np.ascontiguousarray(row_ids, dtype=np.int64)
    rows, K = x.shape
    E, N, _ = w.shape
    Y = np.full((len(ids), N), np.nan)
    grp = np.empty(len(ids), np.int32)
    _check(_load().gdg_oracle_fwd_rows(_ptr(x), _ptr(w), _ptr(o), kind, rows, E, N, K,
                                       _ptr(ids), len(ids), _ptr(Y), _ptr(grp)))
    return Y, grp


def dgrad_rows(G, W, offs, row_ids, kind: int = OFFS_ENDS):
    g, w, o = _bits(G), _bits(W), _offs(offs)
    ids = np.ascontiguousarray(row_ids, dtype=np.int64)
    rows, N = g.shape
    E, _, K = w.shape
    dX = np.full((len(ids), K), np.nan)
    grp = np.empty(len(ids), np.int32)
    _check(_load().gdg_oracle_dgrad_rows(_ptr(g), _ptr(w), _ptr(o), kind, rows, E, N, K,
                                         _ptr(ids), len(ids), _ptr(dX), _ptr(grp)))
    return dX, grp


def wgrad_entries(G, X, offs, E: int, N: int, K: int, flat_ids, kind: int = OFFS_ENDS):
    """dW at flat indices e*N*K + n*K + k."""
    g, x, o = _bits(G), _bits(X), _offs(offs)
    ids = np.ascontiguousarray(flat_ids, dtype=np.int64)
    vals = np.empty(len(ids))
    rows = g.shape[0]
    _check(_load().gdg_oracle_wgrad_entries(_ptr(g), _ptr(x), _ptr(o), kind, rows, E, N, K,
                                            _ptr(ids), len(ids), _ptr(vals)))
    return vals


def wgrad_rows(G, X, offs, E: int, N: int, K: int, pairs, kind: int = OFFS_ENDS):
    """Whole rows dW[e, n, :] for the listed (e, n) pairs -> [len(pairs), K]."""
    g, x, o = _bits(G), _bits(X), _offs(offs)
    ids = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    vals = np.empty((len(ids), K))
    rows = g.shape[0]
    _check(_load().gdg_oracle_wgrad_rows(_ptr(g), _ptr(x), _ptr(o), kind, rows, E, N, K,
                                         _ptr(ids), len(ids), _ptr(vals)))
    return vals
