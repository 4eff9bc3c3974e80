"""Pins of the fp64 oracle against facts fixed outside the oracle itself.

Sources: the computation table and intro paragraph of the "Cake ragged BF16
grouped GEMM (experimental)" docs page (fwd / dgrad / wgrad definitions, group
row ranges from ``offs`` or ``m_indptr``, exact zeros for empty groups) and the
deterministic weight-gradient accumulation section of the MoE grouped GEMM
pull request (``out[e] += G[e].T @ X[e]``).

Each pin is chosen so that a plausible mistake in the oracle (a transposed
operand, a wrong expert, an off-by-one group boundary, a dropped row) fails
at least one of them; ``test_planted_mistakes_are_caught`` shows that by
running mutated copies of the oracle through the same checks.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def f64(t):
    return t.float().double().numpy()


def rand_case(sizes, N, K, seed, lead=0, pad=0, kind=wl.OFFS_ENDS, E=None):
    sizes = np.asarray(sizes)
    E = len(sizes) if E is None else E
    rows = lead + int(sizes.sum()) + pad
    X = wl.normal_bf16((rows, K), 1.0, seed, 1)
    G = wl.normal_bf16((rows, N), 1.0, seed, 2)
    W = wl.normal_bf16((E, N, K), 0.25, seed, 3)
    offs = wl.offsets(sizes, kind, lead)
    return X, G, W, offs


def block_diag_operands(A, offs, kind, E, rows):
    """Dense [rows, E*C] matrix holding row i of A in column block e(i)."""
    st, en = oracle.bounds(offs, kind, E, rows)
    C = A.shape[1]
    out = np.zeros((rows, E * C))
    a = f64(A)
    for e in range(E):
        out[st[e]:en[e], e * C:(e + 1) * C] = a[st[e]:en[e]]
    return out, st, en


# --------------------------------------------------------------------------
# hand-worked fixture
# --------------------------------------------------------------------------

def load_hand():
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("kind", [wl.OFFS_ENDS, wl.OFFS_INDPTR])
def test_hand_example(kind):
    h = load_hand()
    X, G, W = bf(h["X"]), bf(h["G"]), bf(h["W"])
    offs = np.array(h["offs_ends"] if kind == wl.OFFS_ENDS else h["m_indptr"], np.int32)
    sentinel = np.full((h["rows"], h["N"]), 123.0)
    Y = oracle.fwd(X, W, offs, kind, out=sentinel)
    assert np.array_equal(Y[:3], np.array(h["Y_rows_0_2"], float))
    assert np.all(Y[3] == 123.0)          # row 3 belongs to no group
    dX = oracle.dgrad(G, W, offs, kind)
    assert np.array_equal(dX[:3], np.array(h["dX_rows_0_2"], float))
    assert np.all(np.isnan(dX[3]))
    dW = oracle.wgrad(G, X, offs, h["E"], kind)
    assert np.array_equal(dW, np.array(h["dW"], float))
    acc = oracle.wgrad_accumulate(np.full(dW.shape, h["main_grad"]), G, X, offs, h["E"], kind)
    assert np.array_equal(acc, h["main_grad"] + np.array(h["dW"], float))


# --------------------------------------------------------------------------
# identity / permutation weights: Y must equal (a permutation of) the X slice
# --------------------------------------------------------------------------

def perm_weights(E, n, seed):
    rng = np.random.default_rng(seed)
    perms = [rng.permutation(n) for _ in range(E)]
    W = np.zeros((E, n, n), np.float32)
    for e, p in enumerate(perms):
        W[e, np.arange(n), p] = 1.0          # W[e][r, p[r]] = 1
    return perms, bf(W)


def test_identity_weight_reproduces_slice():
    n = 16
    sizes = [3, 0, 5, 1]
    X, G, _, offs = rand_case(sizes, n, n, seed=5)
    W = bf(np.broadcast_to(np.eye(n, dtype=np.float32), (4, n, n)).copy())
    Y = oracle.fwd(X, W, offs)
    dX = oracle.dgrad(G, W, offs)
    assert np.array_equal(Y, f64(X))
    assert np.array_equal(dX, f64(G))


def test_permutation_weight_picks_expert_and_orientation():
    n = 16
    sizes = [4, 2, 0, 6]
    E = len(sizes)
    X, G, _, offs = rand_case(sizes, n, n, seed=6)
    perms, W = perm_weights(E, n, seed=7)
    st, en = oracle.bounds(offs, wl.OFFS_ENDS, E, X.shape[0])
    Y = oracle.fwd(X, W, offs)
    dX = oracle.dgrad(G, W, offs)
    x, g = f64(X), f64(G)
    for e in range(E):
        p = perms[e]
        inv = np.argsort(p)
        for i in range(st[e], en[e]):
            # fwd: Y[i, r] = sum_k X[i, k] W[e][r, k] = X[i, p[r]]
            assert np.array_equal(Y[i], x[i, p])
            # dgrad: dX[i, k] = sum_r G[i, r] W[e][r, k] = G[i, inv[k]]
            assert np.array_equal(dX[i], g[i, inv])


def test_single_row_group_wgrad_is_outer_product():
    sizes = [1, 0, 1]
    X, G, _, offs = rand_case(sizes, 8, 24, seed=8)
    dW = oracle.wgrad(G, X, offs, 3)
    assert np.array_equal(dW[0], np.outer(f64(G)[0], f64(X)[0]))
    assert np.array_equal(dW[2], np.outer(f64(G)[1], f64(X)[1]))
    assert np.array_equal(dW[1], np.zeros((8, 24)))


# --------------------------------------------------------------------------
# brute force: dense block-diagonal matmul (numpy fp64, a library routine)
# --------------------------------------------------------------------------

CASES = [
    dict(sizes=[3, 0, 5, 1], lead=0, pad=0, kind=wl.OFFS_ENDS),
    dict(sizes=[0, 0, 7], lead=0, pad=2, kind=wl.OFFS_ENDS),
    dict(sizes=[6], lead=0, pad=0, kind=wl.OFFS_ENDS),
    dict(sizes=[2, 9, 0, 0, 4], lead=3, pad=1, kind=wl.OFFS_INDPTR),
]


@pytest.mark.parametrize("case", CASES)
def test_block_diagonal_bruteforce(case):
    N, K = 12, 20
    X, G, W, offs = rand_case(case["sizes"], N, K, seed=9, lead=case["lead"],
                              pad=case["pad"], kind=case["kind"])
    E, rows, kind = len(case["sizes"]), X.shape[0], case["kind"]
    Xb, st, en = block_diag_operands(X, offs, kind, E, rows)
    Gb, _, _ = block_diag_operands(G, offs, kind, E, rows)
    w = f64(W)
    Wb_f = np.concatenate([w[e].T for e in range(E)], axis=0)   # [E*K, N]
    Wb_d = np.concatenate([w[e] for e in range(E)], axis=0)     # [E*N, K]
    in_group = np.zeros(rows, bool)
    for e in range(E):
        in_group[st[e]:en[e]] = True

    Y = oracle.fwd(X, W, offs, kind)
    np.testing.assert_allclose(Y[in_group], (Xb @ Wb_f)[in_group], rtol=1e-12, atol=1e-12)
    assert np.all(np.isnan(Y[~in_group]))

    dX = oracle.dgrad(G, W, offs, kind)
    np.testing.assert_allclose(dX[in_group], (Gb @ Wb_d)[in_group], rtol=1e-12, atol=1e-12)
    assert np.all(np.isnan(dX[~in_group]))

    dW = oracle.wgrad(G, X, offs, E, kind)
    full = Gb.T @ Xb                                            # [E*N, E*K]
    for e in range(E):
        np.testing.assert_allclose(dW[e], full[e * N:(e + 1) * N, e * K:(e + 1) * K],
                                   rtol=1e-12, atol=1e-12)


def test_integer_exact_cases_match_bitwise():
    N, K = 32, 48
    sizes = [5, 0, 9, 1]
    E = len(sizes)
    rows = sum(sizes)
    X = wl.integer_bf16((rows, K), -2, 2, seed=1, tag=1)
    G = wl.integer_bf16((rows, N), -2, 2, seed=1, tag=2)
    W = wl.integer_bf16((E, N, K), -2, 2, seed=1, tag=3)
    offs = wl.offsets(sizes)
    Xb, st, en = block_diag_operands(X, offs, wl.OFFS_ENDS, E, rows)
    Gb, _, _ = block_diag_operands(G, offs, wl.OFFS_ENDS, E, rows)
    w = f64(W)
    assert np.array_equal(oracle.fwd(X, W, offs),
                          Xb @ np.concatenate([w[e].T for e in range(E)], axis=0))
    assert np.array_equal(oracle.dgrad(G, W, offs),
                          Gb @ np.concatenate([w[e] for e in range(E)], axis=0))
    dW = oracle.wgrad(G, X, offs, E)
    full = Gb.T @ Xb
    for e in range(E):
        assert np.array_equal(dW[e], full[e * N:(e + 1) * N, e * K:(e + 1) * K])


# --------------------------------------------------------------------------
# exact zeros, adjoint identity, additivity, conventions
# --------------------------------------------------------------------------

def test_empty_groups_give_positive_zero_dW():
    X, G, _, offs = rand_case([0, 4, 0, 0, 3], 8, 16, seed=10)
    dW = oracle.wgrad(G, X, offs, 5)
    for e in (0, 2, 3):
        assert np.all(dW[e] == 0.0) and not np.any(np.signbit(dW[e]))
    assert np.count_nonzero(dW[1]) > 0 and np.count_nonzero(dW[4]) > 0


def test_accumulate_is_main_grad_plus_dW():
    X, G, _, offs = rand_case([0, 4, 3], 8, 16, seed=11)
    mg = wl.normal_fp32((3, 8, 16), 1.0, 11, 4).numpy()
    mg[0, 0, 0] = -0.0
    acc = oracle.wgrad_accumulate(mg, G, X, offs, 3)
    dW = oracle.wgrad(G, X, offs, 3)
    assert np.array_equal(acc, mg.astype(np.float64) + dW)
    assert np.array_equal(acc[0], mg[0].astype(np.float64) + 0.0)
    assert acc[0, 0, 0] == 0.0 and not np.signbit(acc[0, 0, 0])   # -0 + +0 = +0


@pytest.mark.parametrize("case", CASES)
def test_adjoint_identity(case):
    """<X W^T, G> = <G W, X> = <G^T X, W> summed over groups: all equal
    sum_e sum_{i,n,k} g(i,n) x(i,k) w(e,n,k)."""
    N, K = 12, 20
    X, G, W, offs = rand_case(case["sizes"], N, K, seed=12, lead=case["lead"],
                              pad=case["pad"], kind=case["kind"])
    E, rows, kind = len(case["sizes"]), X.shape[0], case["kind"]
    st, en = oracle.bounds(offs, kind, E, rows)
    mask = np.zeros(rows, bool)
    for e in range(E):
        mask[st[e]:en[e]] = True
    Y = oracle.fwd(X, W, offs, kind)
    dX = oracle.dgrad(G, W, offs, kind)
    dW = oracle.wgrad(G, X, offs, E, kind)
    a = np.sum(Y[mask] * f64(G)[mask])
    b = np.sum(dX[mask] * f64(X)[mask])
    c = np.sum(dW * f64(W))
    scale = np.sum(np.abs(Y[mask] * f64(G)[mask]))   # size of the terms summed
    assert scale > 1.0
    assert abs(a - b) <= 1e-12 * scale and abs(a - c) <= 1e-12 * scale


def test_splitting_a_group_is_additive():
    N, K = 8, 16
    X, G, W, _ = rand_case([7, 5], N, K, seed=13)
    merged = wl.offsets([12])
    split = wl.offsets([7, 5])
    W1 = W[:1]
    W2 = torch.cat([W1, W1], dim=0)
    # fwd / dgrad rows do not depend on how a group is cut
    assert np.array_equal(oracle.fwd(X, W1, merged), oracle.fwd(X, W2, split))
    assert np.array_equal(oracle.dgrad(G, W1, merged), oracle.dgrad(G, W2, split))
    dm = oracle.wgrad(G, X, merged, 1)
    ds = oracle.wgrad(G, X, split, 2)
    np.testing.assert_allclose(dm[0], ds[0] + ds[1], rtol=1e-13, atol=1e-13)


def test_offsets_conventions_agree():
    N, K = 8, 16
    X, G, W, ends = rand_case([3, 0, 4], N, K, seed=14)
    indptr = wl.offsets([3, 0, 4], wl.OFFS_INDPTR)
    assert np.array_equal(oracle.fwd(X, W, ends, wl.OFFS_ENDS),
                          oracle.fwd(X, W, indptr, wl.OFFS_INDPTR))
    assert np.array_equal(oracle.wgrad(G, X, ends, 3, wl.OFFS_ENDS),
                          oracle.wgrad(G, X, indptr, 3, wl.OFFS_INDPTR))


@pytest.mark.parametrize("bad", [[3, 2, 7], [-1, 2, 7], [1, 2, 99]])
def test_invalid_offsets_are_rejected(bad):
    X, G, W, _ = rand_case([3, 0, 4], 8, 16, seed=15)
    with pytest.raises(oracle.OracleError):
        oracle.fwd(X, W, np.array(bad, np.int32))
    with pytest.raises(oracle.OracleError):
        oracle.wgrad(G, X, np.array(bad, np.int32), 3)


def test_sampled_forms_equal_full_forms():
    N, K = 12, 20
    X, G, W, offs = rand_case([2, 9, 0, 4], N, K, seed=16, lead=3, pad=2,
                              kind=wl.OFFS_INDPTR)
    E, rows = 4, X.shape[0]
    Y = oracle.fwd(X, W, offs, wl.OFFS_INDPTR)
    dX = oracle.dgrad(G, W, offs, wl.OFFS_INDPTR)
    dW = oracle.wgrad(G, X, offs, E, wl.OFFS_INDPTR)
    ids = np.arange(rows)
    Ys, grp = oracle.fwd_rows(X, W, offs, ids, wl.OFFS_INDPTR)
    dXs, _ = oracle.dgrad_rows(G, W, offs, ids, wl.OFFS_INDPTR)
    inside = grp >= 0
    assert inside.sum() == 15
    assert np.array_equal(Ys[inside], Y[inside]) and np.array_equal(dXs[inside], dX[inside])
    flat = np.random.default_rng(0).choice(dW.size, 200, replace=False)
    vals = oracle.wgrad_entries(G, X, offs, E, N, K, flat, wl.OFFS_INDPTR)
    assert np.array_equal(vals, dW.ravel()[flat])
    pairs = [(e, n) for e in range(E) for n in (0, 5, N - 1)]
    rows_w = oracle.wgrad_rows(G, X, offs, E, N, K, pairs, wl.OFFS_INDPTR)
    assert np.array_equal(rows_w, np.stack([dW[e, n] for e, n in pairs]))


# --------------------------------------------------------------------------
# the pins catch planted mistakes (mutants of the oracle, CPU only)
# --------------------------------------------------------------------------

def _mut_transposed_w(X, W, offs, kind=wl.OFFS_ENDS):
    return oracle.fwd(X, W.transpose(1, 2).contiguous(), offs, kind)


def _mut_wrong_expert(X, W, offs, kind=wl.OFFS_ENDS):
    return oracle.fwd(X, torch.roll(W, 1, dims=0), offs, kind)


def _mut_off_by_one(X, W, offs, kind=wl.OFFS_ENDS):
    o = np.asarray(offs).copy()
    o[0] += 1
    return oracle.fwd(X, W, o, kind)


def test_planted_mistakes_are_caught():
    n = 16
    sizes = [4, 2, 0, 6]
    X, _, _, offs = rand_case(sizes, n, n, seed=17)
    perms, W = perm_weights(len(sizes), n, seed=18)
    st, en = oracle.bounds(offs, wl.OFFS_ENDS, 4, X.shape[0])
    x = f64(X)

    def permutation_pin(fn):
        Y = fn(X, W, offs)
        return all(np.array_equal(Y[i], x[i, perms[e]])
                   for e in range(4) for i in range(st[e], en[e]))

    assert permutation_pin(oracle.fwd)
    for mutant in (_mut_transposed_w, _mut_wrong_expert, _mut_off_by_one):
        assert not permutation_pin(mutant), mutant.__name__
