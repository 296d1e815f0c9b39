"""Pins of the path-composition oracle (oracle/pcomoe.py), no GPU: diagonal
paths reproduce the vanilla layer (computed by the layer oracle's own FFN),
source-grouped execution equals recomputing the expansion per path, a one-hot
closed form fixes which side comes from the source and which from the
target, and the unique-source bookkeeping matches brute force."""
import numpy as np
import pytest
import torch

from aware_moe_expert_gb300.inputs import make_paths
from oracle import moe_oracle as O
from oracle import pcomoe as P


def _layer(seed, T=9, H=12, E=6, I=5):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, H))
    wgu = rng.normal(size=(E, 2 * I, H)) / 3
    wd = rng.normal(size=(E, H, I)) / 3
    return x, wgu, wd


def _routing(T, E, k_max, seed):
    rng = np.random.default_rng(seed)
    k = rng.integers(1, k_max + 1, T)
    idx = np.full((T, k_max), -1, dtype=np.int64)
    w = np.zeros((T, k_max))
    for t in range(T):
        idx[t, :k[t]] = rng.choice(E, k[t], replace=False)
        w[t, :k[t]] = rng.random(k[t])
    return idx, w, k


def test_diagonal_paths_are_the_vanilla_layer():
    x, wgu, wd = _layer(1)
    idx, w, k = _routing(9, 6, 4, 2)
    out, n_exp = P.paths_forward(x, lambda u: wgu[u], lambda u: wd[u], idx, idx, w, k)
    want = np.zeros_like(x)
    for t in range(9):
        for j in range(k[t]):
            want[t] += w[t, j] * O.swiglu_ffn(x[t:t + 1], wgu[idx[t, j]], wd[idx[t, j]])[0]
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)
    assert n_exp == int(k.sum())


def test_source_grouping_equals_per_path_recomputation():
    x, wgu, wd = _layer(3)
    idx, w, k = _routing(9, 6, 5, 4)
    src, tgt, beta = (t.numpy() for t in make_paths(torch.from_numpy(idx).int(),
                                                      torch.from_numpy(w).float()))
    out, n_exp = P.paths_forward(x, lambda u: wgu[u], lambda u: wd[u], src, tgt, beta, k)
    want = np.zeros_like(x)
    for t in range(9):
        for j in range(k[t]):
            z = P.expansion(x[t:t + 1], wgu[src[t, j]])          # recomputed every path
            want[t] += float(beta[t, j]) * (z @ wd[tgt[t, j]].T)[0]
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)
    uniq = sum(len(set(src[t, :k[t]].tolist())) for t in range(9))
    assert n_exp == uniq < int(k.sum())


def test_one_hot_closed_form_source_and_target_roles():
    """Unit u's single neuron reads input a_u (gate) and b_u (up) and writes
    output c_u: a path (i, j) must give beta * silu(x_{a_i}) * x_{b_i} at
    output c_j (expansion from the source, projection from the target)."""
    H, E = 8, 3
    a, b, c = [0, 2, 4], [1, 3, 5], [6, 7, 0]
    wgu = np.zeros((E, 2, H))
    wd = np.zeros((E, H, 1))
    for u in range(E):
        wgu[u, 0, a[u]] = 1.0
        wgu[u, 1, b[u]] = 1.0
        wd[u, c[u], 0] = 1.0
    x = np.arange(1, H + 1, dtype=np.float64)[None, :] / 4
    src = np.array([[0, 0, 2]])
    tgt = np.array([[0, 1, 1]])
    beta = np.array([[0.5, 2.0, -1.0]])
    out, _ = P.paths_forward(x, lambda u: wgu[u], lambda u: wd[u], src, tgt, beta, [3])
    s = lambda g: g / (1 + np.exp(-g))  # noqa: E731
    want = np.zeros(H)
    want[c[0]] += 0.5 * s(x[0, a[0]]) * x[0, b[0]]
    want[c[1]] += 2.0 * s(x[0, a[0]]) * x[0, b[0]]
    want[c[1]] += -1.0 * s(x[0, a[2]]) * x[0, b[2]]
    np.testing.assert_allclose(out[0], want, rtol=1e-14)


def test_unique_sources_brute_force():
    rng = np.random.default_rng(5)
    src = rng.integers(0, 4, (20, 6))
    n = rng.integers(0, 7, 20)
    srcs, n_src, slot = P.unique_sources(src, n)
    for t in range(20):
        seq = src[t, :n[t]].tolist()
        firsts = [v for i, v in enumerate(seq) if v not in seq[:i]]
        assert srcs[t, :n_src[t]].tolist() == firsts
        assert (srcs[t, n_src[t]:] == -1).all()
        for j in range(n[t]):
            assert firsts[slot[t, j]] == seq[j]


def test_path_recipe_shares_every_second_source():
    idx = torch.tensor([[3, 5, 7, 1], [2, 4, -1, -1]], dtype=torch.int32)
    w = torch.rand(2, 4)
    s, t, b = make_paths(idx, w)
    assert s.tolist() == [[3, 3, 7, 7], [2, 2, -1, -1]]
    assert t.tolist() == idx.tolist()
    assert torch.equal(b[0], w[0]) and b[1, 2:].abs().sum() == 0


def test_shared_expert_term_closed_form():
    """The shared expert adds with weight 1 on top of the paths.  One-hot
    shared weights (neuron n reads gate input a_n and up input b_n, writes
    output c_n) make its term the closed form sum_n silu(x_{a_n}) x_{b_n} at
    c_n; with diagonal paths the rest is the vanilla layer (the layer
    oracle's FFN).  Dropping the shared term, or scaling it, fails this."""
    x, wgu, wd = _layer(11, T=5, H=10, E=4, I=3)
    idx, w, k = _routing(5, 4, 3, 12)
    a, b, c = [1, 4, 7], [2, 5, 9], [0, 3, 3]          # two neurons write output 3
    sgu = np.zeros((2 * 3, 10))
    sd = np.zeros((10, 3))
    for n in range(3):
        sgu[n, a[n]] = 1.0
        sgu[3 + n, b[n]] = 1.0
        sd[c[n], n] = 1.0
    out, _ = P.paths_forward(x, lambda u: wgu[u], lambda u: wd[u], idx, idx, w, k,
                             w_shared_gate_up=sgu, w_shared_down=sd)
    vanilla = np.zeros_like(x)
    for t in range(5):
        for j in range(k[t]):
            vanilla[t] += w[t, j] * O.swiglu_ffn(x[t:t + 1], wgu[idx[t, j]], wd[idx[t, j]])[0]
    shared = np.zeros_like(x)
    for t in range(5):
        for n in range(3):
            g = x[t, a[n]]
            shared[t, c[n]] += g / (1.0 + np.exp(-g)) * x[t, b[n]]
    np.testing.assert_allclose(out, vanilla + shared, rtol=1e-12, atol=1e-12)
    assert np.abs(shared).max() > 0.1                  # the term is not negligible here
    assert not np.allclose(out, vanilla + 0.5 * shared, rtol=1e-6, atol=1e-6)


def test_paths_sharing_a_target_sum_before_the_projection():
    """Two paths of one token with the same target j: the projection is
    linear, so sum_i beta_i D_j(U_i(h)) = D_j(sum_i beta_i U_i(h)); with
    one-hot weights both equal the closed form at the target's output."""
    H, E = 8, 3
    a, b, c = [0, 2, 4], [1, 3, 5], [6, 7, 0]
    wgu = np.zeros((E, 2, H))
    wd = np.zeros((E, H, 1))
    for u in range(E):
        wgu[u, 0, a[u]] = 1.0
        wgu[u, 1, b[u]] = 1.0
        wd[u, c[u], 0] = 1.0
    x = np.arange(1, H + 1, dtype=np.float64)[None, :] / 3
    src = np.array([[0, 2, 1]])
    tgt = np.array([[1, 1, 1]])                        # every path projects through unit 1
    beta = np.array([[0.5, -2.0, 0.25]])
    out, n_exp = P.paths_forward(x, lambda u: wgu[u], lambda u: wd[u], src, tgt, beta, [3])
    s = lambda g: g / (1 + np.exp(-g))  # noqa: E731
    want = np.zeros(H)
    want[c[1]] = sum(beta[0, j] * s(x[0, a[src[0, j]]]) * x[0, b[src[0, j]]] for j in range(3))
    np.testing.assert_allclose(out[0], want, rtol=1e-14)
    merged = sum(beta[0, j] * P.expansion(x, wgu[src[0, j]]) for j in range(3))
    np.testing.assert_allclose(out, P.projection(merged, wd[1]), rtol=1e-14)
    assert n_exp == 3
