"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Cases span several tiles with ragged tails: empty groups, one-row groups,
groups that are not multiples of any tile size, row padding before and after
the groups, both offset conventions, dgrad feature tiles and wgrad k tiles
that are only partly inside K, and the split and unsplit wgrad forms.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import (assert_bf16_close, assert_bitwise, assert_fp32_close, group_rows_mask,
                     inputs_on, to64)

pytestmark = pytest.mark.gpu

DEV = "cuda"

SMALL = [
    # name, E, N, K, sizes, lead, pad, kind
    ("tiny", 4, 256, 256, [200, 0, 311, 1], 0, 0, wl.OFFS_ENDS),
    ("ragged", 6, 512, 320, [300, 0, 1, 17, 513, 255], 0, 5, wl.OFFS_ENDS),
    ("indptr_lead", 5, 256, 448, [0, 129, 64, 0, 700], 3, 2, wl.OFFS_INDPTR),
    ("one_group", 1, 768, 192, [1000], 0, 0, wl.OFFS_ENDS),
    ("all_tiny_groups", 40, 256, 128, [i % 4 for i in range(40)], 0, 1, wl.OFFS_ENDS),
    # more than 64 rows per group on average: fwd / dgrad take the 256-row tile
    ("big_groups", 3, 512, 320, [700, 1, 601], 0, 3, wl.OFFS_ENDS),
    # groups longer than 2048 rows: an fp32 weight gradient is reduced in 2048-row chunks
    ("long_groups", 3, 256, 128, [5000, 3, 2100], 0, 0, wl.OFFS_ENDS),
]


def small_case(spec, seed=1):
    name, E, N, K, sizes, lead, pad, kind = spec
    w = wl.Workload(name, E=E, N=N, K=K, ops=(), main_grad_std=1.0)
    return inputs_on(w, DEV, seed=seed, sizes=sizes, kind=kind, pad_rows=pad, lead=lead)


@pytest.mark.parametrize("spec", SMALL, ids=[s[0] for s in SMALL])
def test_fwd_dgrad_match_oracle(cuda_lib, spec):
    h, d = small_case(spec)
    w, kind, rows = h["workload"], h["kind"], h["rows"]
    mask = group_rows_mask(h["offs_np"], kind, w.E, rows)
    sentinel = torch.full((rows, w.N), -7.0, dtype=torch.bfloat16, device=DEV)
    Y = cuda_lib.grouped_det_gemm_fwd(d["X"], d["W"], d["offs"], out=sentinel.clone(),
                                      offs_kind=kind)
    ref = oracle.fwd(h["X"], h["W"], h["offs_np"], kind)
    assert_bf16_close(Y[torch.from_numpy(mask).to(DEV)], ref[mask], "fwd")
    assert torch.all(Y[torch.from_numpy(~mask).to(DEV)] == -7.0), "fwd wrote rows outside groups"

    sentinel = torch.full((rows, w.K), -7.0, dtype=torch.bfloat16, device=DEV)
    dX = cuda_lib.grouped_det_gemm_dgrad(d["G"], d["W"], d["offs"], out=sentinel,
                                         offs_kind=kind)
    ref = oracle.dgrad(h["G"], h["W"], h["offs_np"], kind)
    assert_bf16_close(dX[torch.from_numpy(mask).to(DEV)], ref[mask], "dgrad")
    assert torch.all(dX[torch.from_numpy(~mask).to(DEV)] == -7.0), "dgrad wrote rows outside groups"


@pytest.mark.parametrize("split_rows", [-1, 64, 128, 0])
@pytest.mark.parametrize("spec", SMALL, ids=[s[0] for s in SMALL])
def test_wgrad_matches_oracle(cuda_lib, spec, split_rows):
    h, d = small_case(spec)
    w, kind = h["workload"], h["kind"]
    ref = oracle.wgrad(h["G"], h["X"], h["offs_np"], w.E, kind)
    dW32 = cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out_dtype=torch.float32,
                                           split_rows=split_rows, offs_kind=kind)
    assert_fp32_close(dW32, ref, "wgrad fp32")
    dW16 = cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out_dtype=torch.bfloat16,
                                           split_rows=split_rows, offs_kind=kind)
    assert_bf16_close(dW16, ref, "wgrad bf16")
    empty = [e for e in range(w.E) if h["sizes"][e] == 0]
    for e in empty:
        assert torch.all(dW32[e].view(torch.int32) == 0), "empty group must give +0.0"
        assert torch.all(dW16[e].view(torch.int16) == 0), "empty group must give +0.0"


@pytest.mark.parametrize("split_rows", [-1, 128])
@pytest.mark.parametrize("spec", SMALL[:3], ids=[s[0] for s in SMALL[:3]])
def test_wgrad_accumulate(cuda_lib, spec, split_rows):
    h, d = small_case(spec)
    w, kind = h["workload"], h["kind"]
    mg0 = d["main_grad"].clone()
    mg0[0, 0, :4] = torch.tensor([-0.0, float("nan"), float("inf"), -0.0])
    # fp32: bitwise equal to main_grad.add_(dW) with dW the same call's overwrite result
    dW = cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out_dtype=torch.float32,
                                         split_rows=split_rows, offs_kind=kind)
    fused = mg0.clone()
    cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=fused, accumulate=True,
                                    split_rows=split_rows, offs_kind=kind)
    assert_bitwise(fused, mg0.clone().add_(dW), "fp32 accumulate vs add_")
    ref = oracle.wgrad_accumulate(mg0.cpu(), h["G"], h["X"], h["offs_np"], w.E, kind)
    finite = np.isfinite(ref)
    assert_fp32_close(fused.cpu()[torch.from_numpy(finite)],
                      ref[finite], "fp32 accumulate vs oracle")
    # bf16 main_grad
    mg16 = mg0.to(torch.bfloat16)
    dW16 = cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out_dtype=torch.bfloat16,
                                           split_rows=split_rows, offs_kind=kind)
    fused16 = mg16.clone()
    cuda_lib.grouped_det_gemm_wgrad(d["G"], d["X"], d["offs"], out=fused16, accumulate=True,
                                    split_rows=split_rows, offs_kind=kind)
    assert_bitwise(fused16, mg16.clone().add_(dW16), "bf16 accumulate vs add_")


@pytest.mark.parametrize("sizes", [[37, 0, 1, 30, 64], [300, 333]],
                         ids=["row_tile_128", "row_tile_256"])
def test_integer_exact_bitwise(cuda_lib, sizes):
    """Small-integer operands: every partial sum is exact in fp32 and the results are
    exact in bf16, so every summation order gives the oracle's value exactly.  The two size
    lists put fwd / dgrad on the 128-row and on the 256-row tile (average group size at most
    or above 64 rows)."""
    E, N, K = len(sizes), 256, 192
    rows = sum(sizes) + 3
    X = wl.integer_bf16((rows, K), -2, 2, seed=3, tag=1)
    G = wl.integer_bf16((rows, N), -2, 2, seed=3, tag=2)
    W = wl.integer_bf16((E, N, K), -1, 1, seed=3, tag=3)
    offs = wl.offsets(sizes)
    mask = group_rows_mask(offs, wl.OFFS_ENDS, E, rows)
    o = torch.from_numpy(offs).to(DEV)
    Y = cuda_lib.grouped_det_gemm_fwd(X.to(DEV), W.to(DEV), o)
    dX = cuda_lib.grouped_det_gemm_dgrad(G.to(DEV), W.to(DEV), o)
    for split in (-1, 64):
        dW = cuda_lib.grouped_det_gemm_wgrad(G.to(DEV), X.to(DEV), o, out_dtype=torch.float32,
                                             split_rows=split)
        assert np.array_equal(to64(dW), oracle.wgrad(G, X, offs, E)), f"wgrad split={split}"
    yref = oracle.fwd(X, W, offs)
    dref = oracle.dgrad(G, W, offs)
    assert np.abs(yref[mask]).max() <= 256 and np.abs(dref[mask]).max() <= 256
    assert np.array_equal(to64(Y)[mask], yref[mask])
    assert np.array_equal(to64(dX)[mask], dref[mask])


def test_permutation_weights_exact(cuda_lib):
    """W[e] a permutation matrix: Y and dX rows are exact permutations of X / G rows."""
    n = 256
    sizes = [5, 0, 300, 1]
    E = len(sizes)
    rows = sum(sizes)
    rng = np.random.default_rng(2)
    perms = [rng.permutation(n) for _ in range(E)]
    Wn = np.zeros((E, n, n), np.float32)
    for e, p in enumerate(perms):
        Wn[e, np.arange(n), p] = 1.0
    W = torch.from_numpy(Wn).to(torch.bfloat16)
    X = wl.normal_bf16((rows, n), 1.0, 4, 1)
    G = wl.normal_bf16((rows, n), 1.0, 4, 2)
    offs = wl.offsets(sizes)
    o = torch.from_numpy(offs).to(DEV)
    Y = to64(cuda_lib.grouped_det_gemm_fwd(X.to(DEV), W.to(DEV), o))
    dX = to64(cuda_lib.grouped_det_gemm_dgrad(G.to(DEV), W.to(DEV), o))
    x, g = to64(X), to64(G)
    st, en = oracle.bounds(offs, wl.OFFS_ENDS, E, rows)
    for e in range(E):
        inv = np.argsort(perms[e])
        for i in range(st[e], en[e]):
            assert np.array_equal(Y[i], x[i, perms[e]]), (e, i)
            assert np.array_equal(dX[i], g[i, inv]), (e, i)


def test_rows_zero(cuda_lib):
    E, N, K = 3, 256, 128
    X = torch.empty((0, K), dtype=torch.bfloat16, device=DEV)
    G = torch.empty((0, N), dtype=torch.bfloat16, device=DEV)
    W = torch.randn((E, N, K), device=DEV).to(torch.bfloat16)
    offs = torch.zeros(E, dtype=torch.int32, device=DEV)
    assert cuda_lib.grouped_det_gemm_fwd(X, W, offs).shape == (0, N)
    assert cuda_lib.grouped_det_gemm_dgrad(G, W, offs).shape == (0, K)
    out = torch.full((E, N, K), 3.0, device=DEV)
    out[0, 0, 0] = -0.0
    cuda_lib.grouped_det_gemm_wgrad(G, X, offs, out=out, accumulate=True)
    assert out.view(torch.int32)[0, 0, 0] == torch.tensor(-0.0).view(torch.int32)  # untouched
    assert torch.all(out.view(-1)[1:] == 3.0)
    dW = torch.full((E, N, K), 3.0, device=DEV)
    cuda_lib.grouped_det_gemm_wgrad(G, X, offs, out=dW)
    assert torch.all(dW.view(torch.int32) == 0)
    torch.cuda.synchronize()
    assert cuda_lib.gdg_device_error() == 0
