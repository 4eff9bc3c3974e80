"""Seeded synthetic workloads for the ragged BF16 grouped GEMM.

This module only draws inputs: group sizes from routing simulations and
random bf16 operands.  It holds none of the GEMM's arithmetic, so both the
fp64 oracle (``oracle/``) and the CUDA library's tests and benchmark can use
it without sharing any of the computation under test.

Group layout ("Cake ragged BF16 grouped GEMM (experimental)" docs page, intro
paragraph): groups are consecutive row ranges of the packed activations,
given by an int32 device tensor, either ``offs[E]`` (cumulative ends) or
``m_indptr[E + 1]`` (leading zero).  Rows are packed by expert ascending,
then by token ascending.

Value recipe (the plainest reading of the workload descriptions): every
operand entry is drawn independently from a normal distribution in fp32
with the stated standard deviation and rounded to bf16 (round to nearest
even, by ``torch.Tensor.to``).  ``N(0, 1/sqrt(K))`` is read as standard
deviation ``1/sqrt(K)``; ``main_grad`` stays fp32.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

OFFS_ENDS = 0
OFFS_INDPTR = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    E: int
    N: int
    K: int
    ops: tuple          # which operations the workload exercises
    x_std: float = 1.0
    g_std: float = 1.0
    w_std: float | None = None     # None -> 1/sqrt(K)
    main_grad_std: float | None = None

    @property
    def weight_std(self) -> float:
        return self.w_std if self.w_std is not None else 1.0 / math.sqrt(self.K)


TINY = Workload("tiny", E=4, N=256, K=256,
                ops=("fwd", "dgrad", "wgrad_bf16", "wgrad_fp32", "wgrad_fp32_acc"),
                main_grad_std=1.0)
MIXTRAL = Workload("mixtral", E=8, N=14336, K=4096, ops=("fwd", "dgrad", "wgrad_bf16"))
FINE = Workload("fine_grained", E=128, N=4096, K=7168, ops=("fwd", "dgrad", "wgrad_bf16"))
WGRAD_HEAVY = Workload("wgrad_heavy", E=64, N=1536, K=2048, ops=("wgrad_fp32_acc",),
                       main_grad_std=0.01)
DECODE = Workload("decode", E=256, N=2048, K=7168, ops=("fwd", "dgrad"))

WORKLOADS = {w.name: w for w in (TINY, MIXTRAL, FINE, WGRAD_HEAVY, DECODE)}


def _rng(seed: int, tag: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, tag]))


# --------------------------------------------------------------------------
# group sizes (routing simulations)
# --------------------------------------------------------------------------

def sizes_tiny(seed: int = 0) -> np.ndarray:
    """Fixed ragged split: one empty group, one single-row group."""
    return np.array([200, 0, 311, 1], dtype=np.int64)


def sizes_mixtral(seed: int = 0, tokens: int = 8192, E: int = 8, topk: int = 2) -> np.ndarray:
    """Top-2 of softmax(N(0,1) logits); softmax is monotone, so the top-2 of
    the logits is taken directly.  Ties go to the lower expert index."""
    logits = _rng(seed, 1).standard_normal((tokens, E))
    order = np.argsort(-logits, axis=1, kind="stable")[:, :topk]
    return np.bincount(order.ravel(), minlength=E).astype(np.int64)


def sizes_fine(seed: int = 0, tokens: int = 4096, E: int = 128, topk: int = 8,
               s: float = 1.1) -> np.ndarray:
    """Each token picks ``topk`` distinct experts without replacement with
    probability proportional to rank**-s; ranks are a seeded permutation."""
    rng = _rng(seed, 2)
    rank = rng.permutation(E) + 1
    p = rank.astype(np.float64) ** (-s)
    p /= p.sum()
    counts = np.zeros(E, dtype=np.int64)
    for _ in range(tokens):
        counts[rng.choice(E, size=topk, replace=False, p=p)] += 1
    return counts


def sizes_wgrad_heavy(seed: int = 0, M: int = 65536, E: int = 64, alpha: float = 0.3,
                      n_empty: int = 3, n_one: int = 2, floor_rows: int = 2) -> np.ndarray:
    """Dirichlet(alpha) shares of M rows with ``n_empty`` forced-empty and
    ``n_one`` forced single-row groups (indices drawn from the seed).  Every
    other group gets ``floor_rows`` plus its floored share of the rest; the
    remainder goes by largest fractional part, ties to the lower index."""
    rng = _rng(seed, 3)
    p = rng.dirichlet(alpha * np.ones(E))
    special = rng.choice(E, size=n_empty + n_one, replace=False)
    empty, one = special[:n_empty], special[n_empty:]
    rest = np.setdiff1d(np.arange(E), special)
    sizes = np.zeros(E, dtype=np.int64)
    sizes[one] = 1
    pool = M - n_one - floor_rows * len(rest)
    share = p[rest] / p[rest].sum() * pool
    base = np.floor(share).astype(np.int64)
    frac = share - base
    left = pool - int(base.sum())
    order = sorted(range(len(rest)), key=lambda j: (-frac[j], rest[j]))
    for j in order[:left]:
        base[j] += 1
    sizes[rest] = floor_rows + base
    assert sizes.sum() == M and (sizes[empty] == 0).all()
    return sizes


def sizes_decode(seed: int = 0, tokens: int = 32, E: int = 256, topk: int = 8) -> np.ndarray:
    rng = _rng(seed, 4)
    counts = np.zeros(E, dtype=np.int64)
    for _ in range(tokens):
        counts[rng.choice(E, size=topk, replace=False)] += 1
    return counts


SIZES = {"tiny": sizes_tiny, "mixtral": sizes_mixtral, "fine_grained": sizes_fine,
         "wgrad_heavy": sizes_wgrad_heavy, "decode": sizes_decode}


def offsets(sizes, kind: int = OFFS_ENDS, lead: int = 0) -> np.ndarray:
    """int32 offsets for group sizes: cumulative ends ``offs[E]`` or
    ``m_indptr[E+1]``.  ``lead`` shifts every group down by that many rows
    (rows before the first group belong to no group)."""
    ends = lead + np.cumsum(np.asarray(sizes, dtype=np.int64))
    if kind == OFFS_ENDS:
        out = ends
    else:
        out = np.concatenate([[lead], ends])
    assert out.max(initial=0) < 2**31
    return out.astype(np.int32)


# --------------------------------------------------------------------------
# operand values
# --------------------------------------------------------------------------

def normal_bf16(shape, std: float, seed: int, tag: int, device="cpu",
                chunk_rows: int | None = None) -> torch.Tensor:
    """fp32 N(0, std) draws rounded to bf16.  Large tensors are drawn in
    chunks along dim 0 so the fp32 temporary stays small."""
    gen = torch.Generator(device=device)
    gen.manual_seed((seed * 1000003 + tag) & 0x7FFFFFFFFFFFFFFF)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if out.numel() == 0:
        return out
    if chunk_rows is None:
        chunk_rows = max(1, (1 << 27) // max(1, out[0].numel()))
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        tmp = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=gen,
                          device=device, dtype=torch.float32)
        out[r0:r1].copy_(tmp.mul_(std))
    return out


def normal_fp32(shape, std: float, seed: int, tag: int, device="cpu") -> torch.Tensor:
    gen = torch.Generator(device=device)
    gen.manual_seed((seed * 1000003 + tag) & 0x7FFFFFFFFFFFFFFF)
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).mul_(std)


def make_inputs(w: Workload, seed: int = 0, device="cpu", sizes=None,
                kind: int = OFFS_ENDS, pad_rows: int = 0, lead: int = 0,
                need=("X", "W", "G", "main_grad")) -> dict:
    """All operands of one workload: X[rows,K], G[rows,N], W[E,N,K] bf16,
    main_grad[E,N,K] fp32 and the int32 offsets (host numpy and device)."""
    if sizes is None:
        sizes = SIZES[w.name](seed)
    sizes = np.asarray(sizes, dtype=np.int64)
    rows = lead + int(sizes.sum()) + pad_rows
    d = {"workload": w, "sizes": sizes, "rows": rows, "kind": kind,
         "offs_np": offsets(sizes, kind, lead)}
    d["offs"] = torch.from_numpy(d["offs_np"]).to(device)
    if "X" in need:
        d["X"] = normal_bf16((rows, w.K), w.x_std, seed, 11, device)
    if "G" in need:
        d["G"] = normal_bf16((rows, w.N), w.g_std, seed, 12, device)
    if "W" in need:
        d["W"] = normal_bf16((w.E, w.N, w.K), w.weight_std, seed, 13, device)
    if "main_grad" in need and w.main_grad_std is not None:
        d["main_grad"] = normal_fp32((w.E, w.N, w.K), w.main_grad_std, seed, 14, device)
    return d


def integer_bf16(shape, lo: int, hi: int, seed: int, tag: int) -> torch.Tensor:
    """Small integers in [lo, hi], exactly representable in bf16."""
    rng = _rng(seed, 100 + tag)
    return torch.from_numpy(rng.integers(lo, hi + 1, size=shape).astype(np.float32)).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU tensor as uint16 (no arithmetic)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
