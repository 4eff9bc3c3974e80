"""Full-size parity: the Mixtral-style, fine-grained, wgrad-heavy and decode-sized workloads at
their real sizes (seed 0, the inputs bench.py uses), run through the same calls bench.py times,
checked against the fp64 oracle on outputs it can compute one by one.

Every group is checked, not a few picked ones:

* fwd / dgrad: every row within 128 rows of a group boundary (the first and the last 128 rows of
  every group, so every row of a group of at most 256 rows) plus 1024 rows drawn at random from
  the whole packed range;
* wgrad: 4096 random dW entries (n, k) of every group, plus every entry of dW for the two
  largest groups; an empty group must give exactly +0.0 (overwrite) or leave main_grad's bits
  unchanged (accumulate).

The oracle computes each sampled output from a one-group sub-problem made of that group's rows
and weights, copied to the host; the GPU outputs come from the full-size launch.  Tolerances are
the suite's: bf16 outputs |err| <= 1e-2 |ref| + 1e-2 rms, fp32 weight gradients |err| <= 1e-4
rms, rms over the sampled reference values of the tensor.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import BF16_REL, BF16_RMS, FP32_RMS, bits, to64

pytestmark = pytest.mark.gpu

DEV = "cuda"
EDGE = 128              # rows checked at each end of every group
RANDOM_ROWS = 1024      # extra rows drawn from the whole packed range
DW_ENTRIES = 4096       # random dW entries per group
FULL_DW_GROUPS = 2      # largest groups whose whole dW is checked


def edge_rows(m):
    """Local row indices within EDGE rows of either end of a group of m rows."""
    if m <= 2 * EDGE:
        return np.arange(m, dtype=np.int64)
    return np.concatenate([np.arange(EDGE), np.arange(m - EDGE, m)]).astype(np.int64)


def rows_to_check(sizes, rng):
    """{group: sorted local row ids}: every group's edge rows plus RANDOM_ROWS random rows."""
    st = np.concatenate([[0], np.cumsum(sizes)[:-1]])
    M = int(np.sum(sizes))
    picked = {int(e): set(edge_rows(int(sizes[e])).tolist()) for e in np.nonzero(sizes)[0]}
    ends = np.cumsum(sizes)
    for r in rng.choice(M, size=min(M, RANDOM_ROWS), replace=False):
        e = int(np.searchsorted(ends, r, side="right"))
        picked[e].add(int(r - st[e]))
    return {e: np.array(sorted(v), dtype=np.int64) for e, v in picked.items()}


def rms_of(ref):
    return float(np.sqrt(np.mean(ref * ref)))


def close_bf16(gpu, ref, what, rms=None):
    rms = rms_of(ref) if rms is None else rms
    bad = ~(np.abs(gpu - ref) <= BF16_REL * np.abs(ref) + BF16_RMS * rms)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance"


def close_fp32(gpu, ref, what, rms=None):
    rms = rms_of(ref) if rms is None else rms
    bad = ~(np.abs(gpu - ref) <= FP32_RMS * rms)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside 1e-4 rms"


@pytest.mark.parametrize("name", ["mixtral", "fine_grained", "wgrad_heavy", "decode"])
def test_full_size_every_group(cuda_lib, name):
    w = wl.WORKLOADS[name]
    d = wl.make_inputs(w, seed=0, device=DEV)
    sizes, offs = d["sizes"], d["offs"]
    st = np.concatenate([[0], np.cumsum(sizes)[:-1]])
    rng = np.random.default_rng(11)
    gpu = {}
    if "fwd" in w.ops:
        gpu["Y"] = cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], offs)
        gpu["dX"] = cuda_lib.grouped_det_gemm_dgrad(d["G"], d["W"], offs)
    acc = "wgrad_fp32_acc" in w.ops
    if acc:
        out = d["main_grad"].clone()
        cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], offs, out=out, accumulate=True)
        gpu["dW"] = out
    elif "wgrad_bf16" in w.ops:
        gpu["dW"] = cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], offs)
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0

    if "Y" in gpu:
        y_got, y_ref, dx_got, dx_ref = [], [], [], []
        for e, ids in rows_to_check(sizes, rng).items():
            s, m = int(st[e]), int(sizes[e])
            one = np.array([m], dtype=np.int32)      # the group as a one-group problem
            We = d["W"][e:e + 1].cpu()
            gid = torch.from_numpy(s + ids).to(DEV)
            ref, _ = oracle.fwd_rows(d["X"][s:s + m].cpu(), We, one, ids)
            y_got.append(to64(gpu["Y"][gid])), y_ref.append(ref)
            ref, _ = oracle.dgrad_rows(d["G"][s:s + m].cpu(), We, one, ids)
            dx_got.append(to64(gpu["dX"][gid])), dx_ref.append(ref)
        n_rows = sum(len(v) for v in y_ref)
        assert n_rows >= min(int(np.sum(sizes)), RANDOM_ROWS)
        close_bf16(np.concatenate(y_got), np.concatenate(y_ref), f"{name} fwd ({n_rows} rows)")
        close_bf16(np.concatenate(dx_got), np.concatenate(dx_ref), f"{name} dgrad ({n_rows} rows)")

    if "dW" in gpu:
        NK = w.N * w.K
        largest = set(int(e) for e in np.argsort(-sizes, kind="stable")[:FULL_DW_GROUPS])
        got_s, ref_s = [], []                       # sampled entries, all groups
        full_got, full_ref = [], []                 # whole dW of the largest groups
        for e in range(w.E):
            s, m = int(st[e]), int(sizes[e])
            one = np.array([m], dtype=np.int32)
            Ge, Xe = d["G"][s:s + m].cpu(), d["X"][s:s + m].cpu()
            flat = np.sort(rng.choice(NK, size=DW_ENTRIES, replace=False)).astype(np.int64)
            ref = oracle.wgrad_entries(Ge, Xe, one, 1, w.N, w.K, flat) if m else np.zeros(DW_ENTRIES)
            got = to64(gpu["dW"][e].reshape(-1)[torch.from_numpy(flat).to(DEV)])
            if acc:
                ref = ref + to64(d["main_grad"][e].reshape(-1)[torch.from_numpy(flat).to(DEV)])
            got_s.append(got), ref_s.append(ref)
            if e in largest:
                ref = oracle.wgrad(Ge, Xe, one, 1)[0]
                if acc:
                    ref = ref + to64(d["main_grad"][e])
                full_got.append(to64(gpu["dW"][e]).ravel()), full_ref.append(ref.ravel())
        check = close_fp32 if acc else close_bf16
        # Entries drawn uniformly from every group estimate the rms of the whole tensor; the
        # whole-dW check of the largest groups uses that rms too (their own is larger).
        rms_all = rms_of(np.concatenate(ref_s))
        check(np.concatenate(got_s), np.concatenate(ref_s), f"{name} wgrad sampled entries",
              rms_all)
        check(np.concatenate(full_got), np.concatenate(full_ref),
              f"{name} wgrad, whole dW of groups {sorted(largest)}", rms_all)
        for e in np.nonzero(sizes == 0)[0]:
            if acc:
                assert torch.equal(bits(gpu["dW"][int(e)]), bits(d["main_grad"][int(e)])), \
                    f"{name}: empty group {e} changed main_grad"
            else:
                assert torch.all(bits(gpu["dW"][int(e)]) == 0), f"{name}: empty group {e} not +0.0"
