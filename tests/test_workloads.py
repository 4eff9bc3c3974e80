"""The seeded synthetic inputs against the configurations they stand for (CPU only): group-size
recipes (token counts, top-k, forced empty / one-row groups, skew), value distributions
(X, G ~ N(0, 1), W ~ N(0, 1/sqrt(K)) as a standard deviation, main_grad ~ N(0, std)), bf16
rounding of the draws, the offsets conventions and seed reproducibility."""
import numpy as np
import pytest
import torch

import workloads as wl


def test_tiny_sizes_are_the_stated_split():
    assert wl.SIZES["tiny"](0).tolist() == [200, 0, 311, 1]
    assert (wl.TINY.E, wl.TINY.N, wl.TINY.K) == (4, 256, 256)


def test_mixtral_routing_is_top2_of_8192_tokens_over_8_experts():
    s = wl.SIZES["mixtral"](0)
    assert len(s) == 8 and s.sum() == 8192 * 2
    assert s.min() > 0 and s.max() / s.min() < 1.2          # mildly imbalanced
    assert (wl.MIXTRAL.N, wl.MIXTRAL.K) == (14336, 4096)


def test_fine_grained_routing_is_zipf_top8_of_4096_tokens():
    s = wl.SIZES["fine_grained"](0)
    assert len(s) == 128 and s.sum() == 4096 * 8
    assert s.max() <= 4096                                   # 8 distinct experts per token
    assert s.max() > 10 * np.median(s)                       # Zipf-skewed popularity
    assert np.any(s % 128 != 0)                              # non-tile-multiple groups
    assert (wl.FINE.N, wl.FINE.K) == (4096, 7168)


def test_wgrad_heavy_has_3_empty_and_2_one_row_groups_summing_to_65536():
    for seed in range(4):
        s = wl.SIZES["wgrad_heavy"](seed)
        assert len(s) == 64 and s.sum() == 65536
        assert (s == 0).sum() == 3 and (s == 1).sum() == 2
        assert s.max() > 4 * 65536 / 64                      # Dirichlet(0.3): a few dominant groups


def test_decode_routing_is_top8_of_32_tokens_over_256_experts():
    s = wl.SIZES["decode"](0)
    assert len(s) == 256 and s.sum() == 32 * 8
    assert s.max() <= 32 and (s == 0).sum() > 64             # most groups 0-3 rows
    assert np.mean(s <= 3) > 0.95


@pytest.mark.parametrize("kind", [wl.OFFS_ENDS, wl.OFFS_INDPTR])
def test_offsets_conventions(kind):
    sizes = np.array([3, 0, 5, 1])
    o = wl.offsets(sizes, kind=kind, lead=2)
    assert o.dtype == np.int32
    if kind == wl.OFFS_ENDS:
        assert o.tolist() == [5, 5, 10, 11]
    else:
        assert o.tolist() == [2, 5, 5, 10, 11]


def test_value_distributions_and_bf16_rounding():
    w = wl.Workload("dist", E=2, N=512, K=1024, ops=(), main_grad_std=0.01)
    d = wl.make_inputs(w, seed=0, device="cpu", sizes=[3000, 1000])
    for name in ("X", "G"):
        t = d[name].float()
        assert d[name].dtype == torch.bfloat16
        assert abs(t.mean().item()) < 0.01 and abs(t.std().item() - 1.0) < 0.01, name
    wstd = d["W"].float().std().item()
    assert abs(wstd - 1.0 / np.sqrt(w.K)) < 0.02 / np.sqrt(w.K)      # std, not variance
    assert d["main_grad"].dtype == torch.float32
    assert abs(d["main_grad"].std().item() - 0.01) < 0.001
    # bf16 values are the round-to-nearest-even of fp32 draws: re-rounding changes nothing
    x = d["X"]
    assert torch.equal(x.float().to(torch.bfloat16).view(torch.int16), x.view(torch.int16))


def test_seeded_inputs_reproduce_and_seeds_differ():
    w = wl.TINY
    a = wl.make_inputs(w, seed=3, device="cpu")
    b = wl.make_inputs(w, seed=3, device="cpu")
    c = wl.make_inputs(w, seed=4, device="cpu")
    for k in ("X", "G", "W"):
        assert torch.equal(a[k].view(torch.int16), b[k].view(torch.int16)), k
        assert not torch.equal(a[k].view(torch.int16), c[k].view(torch.int16)), k
    assert np.array_equal(wl.SIZES["fine_grained"](1), wl.SIZES["fine_grained"](1))
    assert not np.array_equal(wl.SIZES["fine_grained"](1), wl.SIZES["fine_grained"](2))
