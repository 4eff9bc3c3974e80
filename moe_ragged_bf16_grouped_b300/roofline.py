"""Algorithmic cost of one grouped GEMM call, for rooflines (measurement only: none of the
GEMM's arithmetic is here).

FLOPs count the real rows of every group, 2 M N K with M the summed group sizes.  Bytes are what
the operation must move at least once: fwd / dgrad read the packed rows and the weights of the
non-empty experts and write the packed outputs, 2 (M K + E_ne N K + M N) for both (fwd reads
M K and writes M N, dgrad reads M N and writes M K); wgrad reads G and X and
writes dW, 2 (M K + M N) + E N K s_out, plus E N K s_out read again when it accumulates into an
existing output.  The combined roofline is t_roof = max(FLOPs / P, bytes / BW).
"""
from __future__ import annotations

import numpy as np

NOMINAL_BF16_TFLOPS = 2250.0     # dense BF16 tensor peak of a B300, nominal
NOMINAL_HBM_GBS = 8000.0         # HBM3e bandwidth of a B300, nominal (about 7.7-8 TB/s)


def op_cost(op: str, sizes, N: int, K: int, out_esize: int = 2, accumulate: bool = False):
    """(flops, bytes, weight_bytes) of one call; weight_bytes is the non-empty experts' W."""
    sizes = np.asarray(sizes, dtype=np.int64)
    M = int(sizes.sum())
    E = len(sizes)
    e_ne = int(np.count_nonzero(sizes))
    flops = 2.0 * M * N * K
    if op == "wgrad":
        nbytes = 2 * (M * K + M * N) + E * N * K * out_esize * (2 if accumulate else 1)
        wbytes = 0
    else:
        # fwd reads X [M, K] and writes Y [M, N]; dgrad reads G [M, N] and writes dX [M, K]
        nbytes = 2 * (M * K + e_ne * N * K + M * N)
        wbytes = 2 * e_ne * N * K
    return flops, float(nbytes), float(wbytes)


def roofline(ms: float, flops: float, nbytes: float, peak_tflops: float, peak_gbs: float):
    """t_roof against the given peaks and the fraction of it reached in ms."""
    t_f = flops / (peak_tflops * 1e12) * 1e3
    t_b = nbytes / (peak_gbs * 1e9) * 1e3
    t_roof = max(t_f, t_b)
    return {"t_roof_ms": t_roof, "bound": "tensor" if t_f >= t_b else "hbm",
            "frac_of_roof": t_roof / ms if ms > 0 else None}
