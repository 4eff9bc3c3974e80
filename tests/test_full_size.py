"""Full-size parity: the Mixtral-style, fine-grained, wgrad-heavy and decode-sized workloads at
their real sizes (seed 0, the inputs bench.py uses), run through the same calls bench.py times,
checked on sampled outputs against the fp64 oracle.

For each workload a few groups are picked (the smallest and largest non-empty group, the median
one, a one-row group if there is one).  The oracle computes the sampled outputs of a one-group
sub-problem made of that group's rows and weights, copied to the host; the GPU outputs come from
the full-size launch.  Tolerances are the suite's: bf16 outputs |err| <= 1e-2 |ref| + 1e-2 rms,
fp32 weight gradients |err| <= 1e-4 rms, rms over the sampled reference values.  Empty groups
must give exactly +0.0 (overwrite) or leave main_grad's bits unchanged (accumulate).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import BF16_REL, BF16_RMS, FP32_RMS, bits, to64

pytestmark = pytest.mark.gpu

DEV = "cuda"
ROWS_PER_GROUP = 24     # sampled Y / dX rows per picked group
WROWS_PER_GROUP = 12    # sampled dW rows (e, n, all k) per picked group


def pick_groups(sizes):
    nz = np.nonzero(sizes)[0]
    order = nz[np.argsort(sizes[nz], kind="stable")]
    picks = {int(order[0]), int(order[-1]), int(order[len(order) // 2])}
    ones = [int(e) for e in nz if sizes[e] == 1]
    if ones:
        picks.add(ones[0])
    return sorted(picks)


def sample_rows(m, rng):
    ids = set(range(min(4, m))) | set(range(max(0, m - 4), m))
    extra = rng.choice(m, size=min(m, ROWS_PER_GROUP), replace=False)
    ids |= set(int(i) for i in extra)
    return np.array(sorted(ids)[:ROWS_PER_GROUP + 8], dtype=np.int64)


def close_bf16(gpu, ref, what):
    rms = float(np.sqrt(np.mean(ref * ref)))
    bad = ~(np.abs(gpu - ref) <= BF16_REL * np.abs(ref) + BF16_RMS * rms)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance"


def close_fp32(gpu, ref, what):
    rms = float(np.sqrt(np.mean(ref * ref)))
    bad = ~(np.abs(gpu - ref) <= FP32_RMS * rms)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside 1e-4 rms"


@pytest.mark.parametrize("name", ["mixtral", "fine_grained", "wgrad_heavy", "decode"])
def test_full_size_sampled(cuda_lib, name):
    w = wl.WORKLOADS[name]
    d = wl.make_inputs(w, seed=0, device=DEV)
    sizes, offs = d["sizes"], d["offs"]
    st = np.concatenate([[0], np.cumsum(sizes)[:-1]])
    rng = np.random.default_rng(11)
    gpu = {}
    if "fwd" in w.ops:
        gpu["Y"] = to64(cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], offs))
        gpu["dX"] = to64(cuda_lib.grouped_det_gemm_dgrad(d["G"], d["W"], offs))
    acc = "wgrad_fp32_acc" in w.ops
    if acc:
        out = d["main_grad"].clone()
        cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], offs, out=out, accumulate=True)
        gpu["dW"] = out
    elif "wgrad_bf16" in w.ops:
        gpu["dW"] = cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], offs)
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0

    y_got, y_ref, dx_got, dx_ref, dw_got, dw_ref = [], [], [], [], [], []
    for e in pick_groups(sizes):
        s, m = int(st[e]), int(sizes[e])
        one = np.array([m], dtype=np.int32)          # the group as a one-group problem
        Xe = d["X"][s:s + m].cpu()
        Ge = d["G"][s:s + m].cpu()
        if "Y" in gpu:
            We = d["W"][e:e + 1].cpu()
            ids = sample_rows(m, rng)
            ref, _ = oracle.fwd_rows(Xe, We, one, ids)
            y_got.append(gpu["Y"][s + ids]), y_ref.append(ref)
            ref, _ = oracle.dgrad_rows(Ge, We, one, ids)
            dx_got.append(gpu["dX"][s + ids]), dx_ref.append(ref)
        if "dW" in gpu:
            ns = np.sort(rng.choice(w.N, size=WROWS_PER_GROUP, replace=False))
            pairs = np.stack([np.zeros_like(ns), ns], 1)
            ref = oracle.wgrad_rows(Ge, Xe, one, 1, w.N, w.K, pairs)
            got = to64(gpu["dW"][e, torch.from_numpy(ns).to(DEV)])
            if acc:
                ref = ref + to64(d["main_grad"][e, torch.from_numpy(ns).to(DEV)])
            dw_got.append(got), dw_ref.append(ref)
    if y_got:
        close_bf16(np.concatenate(y_got), np.concatenate(y_ref), f"{name} fwd")
        close_bf16(np.concatenate(dx_got), np.concatenate(dx_ref), f"{name} dgrad")
    if dw_got:
        check = close_fp32 if acc else close_bf16
        check(np.concatenate(dw_got), np.concatenate(dw_ref), f"{name} wgrad")
        for e in np.nonzero(sizes == 0)[0][:4]:
            if acc:
                assert torch.equal(bits(gpu["dW"][int(e)]), bits(d["main_grad"][int(e)])), \
                    f"{name}: empty group {e} changed main_grad"
            else:
                assert torch.all(bits(gpu["dW"][int(e)]) == 0), f"{name}: empty group {e} not +0.0"
