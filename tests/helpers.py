"""Shared helpers of the GPU tests: tolerance checks against the fp64 oracle.

Tolerances (stated for this path): bf16 outputs |gpu - ref| <= 1e-2 |ref| +
1e-2 rms(ref); fp32 weight gradients |gpu - ref| <= 1e-4 rms(ref), rms over
the rows that belong to a group (fwd / dgrad) or over all of dW (wgrad).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as wl

BF16_REL, BF16_RMS = 1e-2, 1e-2
FP32_RMS = 1e-4


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().double().cpu().numpy()


def group_rows_mask(offs_np, kind, E, rows) -> np.ndarray:
    st, en = oracle.bounds(offs_np, kind, E, rows)
    m = np.zeros(rows, bool)
    for e in range(E):
        m[st[e]:en[e]] = True
    return m


def assert_bf16_close(gpu: torch.Tensor, ref: np.ndarray, what: str = ""):
    g = to64(gpu)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    if ref.size == 0:
        return
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(g - ref)
    bound = BF16_REL * np.abs(ref) + BF16_RMS * rms
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:8]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside tolerance (rms {rms:.4g}); "
            f"first {idx.tolist()} gpu {g[bad][:8]} ref {ref[bad][:8]}")


def assert_fp32_close(gpu: torch.Tensor, ref: np.ndarray, what: str = ""):
    g = to64(gpu)
    assert g.shape == ref.shape
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = np.abs(g - ref)
    bad = ~(err <= FP32_RMS * rms)
    if bad.any():
        idx = np.argwhere(bad)[:8]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside 1e-4*rms (rms {rms:.4g}); "
            f"first {idx.tolist()} gpu {g[bad][:8]} ref {ref[bad][:8]}")


def bits(t: torch.Tensor) -> torch.Tensor:
    """Raw bits for bitwise comparisons (NaN-safe)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16)
    if t.dtype == torch.float32:
        return t.view(torch.int32)
    return t


def assert_bitwise(a: torch.Tensor, b: torch.Tensor, what: str = ""):
    ba, bb = bits(a), bits(b)
    if not torch.equal(ba, bb):
        diff = (ba != bb).nonzero()[:8].tolist()
        raise AssertionError(f"{what}: not bitwise equal at {diff}")


def inputs_on(w: wl.Workload, device, seed=0, **kw):
    """Generate on the CPU (small shapes) and copy to the device; keep both."""
    d = wl.make_inputs(w, seed=seed, device="cpu", **kw)
    dev = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    return d, dev
