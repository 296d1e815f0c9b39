"""Pins of the proxy-router (CG) oracle against closed forms, brute force and
an independent formulation (MoE-Prism, arXiv 2510.19366, §III-B2,
"Training-Free Proxy Gating").  CPU only."""
import math

import numpy as np
import pytest

from oracle import moe_oracle as O
from oracle import cg_router as CG


def _split_layer(rng, n_experts, n_sub, I_sub, H):
    """Random fp64 weights of a split layer: per unit [2 I_sub, H] and [H, I_sub]."""
    E_r = n_experts * n_sub
    wgu = rng.standard_normal((E_r, 2 * I_sub, H)) / math.sqrt(H)
    wd = rng.standard_normal((E_r, H, I_sub)) / math.sqrt(n_sub * I_sub)
    return wgu, wd


def test_full_allocation_reproduces_unsplit_top_m_moe():
    """kappa_j = N for every selected expert: all N sub-experts of each of the
    top-m experts run with the expert's weight, which must equal the
    monolithic top-m MoE written out directly (Eq. (3): an expert is the sum
    of its sub-experts)."""
    rng = np.random.default_rng(1)
    T, H, E, N, I_sub, m = 6, 8, 4, 3, 4, 2
    spec = O.LayerSpec(T=T, H=H, n_experts=E, n_sub=N, I_sub=I_sub, k_max=m * N, renorm=True)
    x = rng.standard_normal((T, H))
    rw = rng.standard_normal((E, H))
    wgu, wd = _split_layer(rng, E, N, I_sub, H)
    G = np.tile(np.arange(2, dtype=np.int32), (E * N, 1))
    kappa = CG.default_kappa(m * N, m, N)
    k = np.full(T, m * N)
    got = CG.layer_forward_cg(spec, x, rw, wgu, wd, G, m, kappa, k)["out"]
    # independent: monolithic experts, dense loop over the top-m
    want = np.zeros((T, H))
    for t in range(T):
        L = rw @ x[t]
        top = sorted(range(E), key=lambda e: (-L[e], e))[:m]
        p = np.exp(L - L.max())
        p = p / p.sum()
        wsum = sum(p[e] for e in top)
        for e in top:
            Wg = np.concatenate([wgu[e * N + n][:I_sub] for n in range(N)])   # [C, H]
            Wu = np.concatenate([wgu[e * N + n][I_sub:] for n in range(N)])
            Wd = np.concatenate([wd[e * N + n] for n in range(N)], axis=1)     # [H, C]
            g, u = Wg @ x[t], Wu @ x[t]
            a = g / (1.0 + np.exp(-g)) * u
            want[t] += (p[e] / wsum) * (Wd @ a)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_proxy_score_closed_form_on_one_hot_rows():
    """Gate row c of sub-expert n = e_{a}, up row c = e_{b}: the neuron's
    activation is SiLU(x_a) * x_b, so s_n is the mean of |SiLU(x_a) x_b| over
    the gate neurons (gate and up swapped, a missing |.|, or the up rows read
    from the wrong offset all change the value)."""
    H, I_sub, r = 6, 5, 2
    x = np.array([0.7, -1.3, 2.1, -0.4, 0.9, -2.2])
    units, G = [], []
    # (a's, b's) of the two gate neurons; SiLU(x_a) x_b is negative for one
    # neuron of each sub-expert, so the |.| matters
    picks = [((0, 1), (1, 5)), ((3, 4), (2, 0))]
    for n, (aa, bb) in enumerate(picks):
        W = np.zeros((2 * I_sub, H))
        g_local = np.array([1, 3]) if n == 0 else np.array([4, 0])
        for c, a, b in zip(g_local, aa, bb):
            W[c, a] = 1.0
            W[I_sub + c, b] = 1.0
        units.append(W)
        G.append(g_local)
    got = CG.proxy_scores(x, units, G)
    silu = lambda v: v / (1.0 + math.exp(-v))
    want = [np.mean([abs(silu(x[a]) * x[b]) for a, b in zip(aa, bb)]) for aa, bb in picks]
    np.testing.assert_allclose(got, want, rtol=1e-15)
    assert r == 2


def test_selection_equals_brute_force_sort():
    """Given expert logits and proxy scores (with ties, -0/+0 and a NaN), the
    chosen units are: expert order by logit, then the kappa_j best
    sub-experts by score, ties to the lower index, NaN last."""
    rng = np.random.default_rng(7)
    T, E, N, m, k_max = 40, 6, 4, 3, 9
    spec = O.LayerSpec(T=T, H=8, n_experts=E, n_sub=N, I_sub=4, k_max=k_max)
    Le = rng.integers(-3, 3, size=(T, E)).astype(np.float32)        # many expert ties
    P = rng.integers(0, 4, size=(T, m, N)).astype(np.float32)       # many score ties
    P[0, 0, :] = [0.0, -0.0, 0.0, -0.0]
    P[1, 1, 2] = np.nan
    kappa = rng.integers(0, N + 1, size=(k_max + 1, m))
    for kk in range(k_max + 1):                                      # valid rows summing to kk
        row = np.zeros(m, dtype=np.int64)
        left = kk
        for j in rng.permutation(m):
            row[j] = min(N, left) if j == m - 1 else rng.integers(0, min(N, left) + 1)
            left -= row[j]
        while left > 0:
            j = int(np.argmin(row))
            add = min(N - row[j], left)
            row[j] += add
            left -= add
        kappa[kk] = row
    k = rng.integers(1, k_max + 1, size=T)
    res = CG.route_cg(spec, None, None, None, None, m, kappa, k, expert_logits=Le, proxy=P)
    for t in range(T):
        experts = sorted(range(E), key=lambda e: (-float(Le[t, e]), e))[:m]
        want = []
        for j, e in enumerate(experts):
            key = lambda n: (1 if math.isnan(P[t, j, n]) else 0,
                             0.0 if math.isnan(P[t, j, n]) else -float(P[t, j, n]), n)
            want += [e * N + n for n in sorted(range(N), key=key)[: kappa[k[t]][j]]]
        got = res["topk_idx"][t]
        assert list(got[: len(want)]) == want, t
        assert (got[len(want):] == -1).all()
        assert list(res["expert_idx"][t]) == experts


def test_selected_units_inherit_their_expert_weight():
    rng = np.random.default_rng(3)
    T, E, N, m = 12, 5, 2, 3
    spec = O.LayerSpec(T=T, H=8, n_experts=E, n_sub=N, I_sub=4, k_max=m * N, renorm=True,
                       route_scale=2.5)
    Le = rng.standard_normal((T, E)).astype(np.float32)
    P = rng.random((T, m, N)).astype(np.float32)
    kappa = CG.default_kappa(m * N, m, N)
    k = rng.integers(1, m * N + 1, size=T)
    res = CG.route_cg(spec, None, None, None, None, m, kappa, k, expert_logits=Le, proxy=P)
    for t in range(T):
        np.testing.assert_allclose(res["expert_w"][t].sum(), 2.5, rtol=1e-12)
        for s in range(int(k[t])):
            e = res["topk_idx"][t, s] // N
            j = list(res["expert_idx"][t]).index(e)
            assert res["topk_w"][t, s] == res["expert_w"][t, j]


def test_gate_neurons_equal_explicit_pair_count():
    """G_n from C_co = B^T B equals counting, for each pair of neurons of the
    same sub-expert, the calibration tokens where both are among the k_a
    largest |A| (self-pairs excluded), and keeping the r best."""
    rng = np.random.default_rng(11)
    Bn, n_sub, I_sub, k_a, r = 9, 3, 4, 5, 2
    C = n_sub * I_sub
    A = rng.integers(-4, 5, size=(Bn, C)).astype(np.float64)   # |A| ties on purpose
    got = CG.gate_neurons(A, n_sub, k_a, r)
    active = []
    for t in range(Bn):
        order = sorted(range(C), key=lambda c: (-abs(A[t, c]), c))
        active.append(set(order[:k_a]))
    for n in range(n_sub):
        S = range(n * I_sub, (n + 1) * I_sub)
        score = {}
        for i in S:
            score[i] = sum(1 for t in range(Bn) for j in S if j != i
                           and i in active[t] and j in active[t])
        best = sorted(S, key=lambda i: (-score[i], i))[:r]
        assert list(got[n]) == [i - n * I_sub for i in best]


@pytest.mark.parametrize("k_max,m,N", [(8, 2, 4), (16, 8, 2), (6, 3, 2), (5, 4, 3)])
def test_default_kappa_is_a_valid_allocation(k_max, m, N):
    K = CG.default_kappa(k_max, m, N)
    for k in range(k_max + 1):
        assert K[k].sum() == k
        assert (K[k] >= 0).all() and (K[k] <= N).all()
        assert (np.diff(K[k]) <= 0).all()          # higher-ranked experts first
        assert K[k].max() - K[k].min() <= 1        # as even as possible


def test_invalid_allocation_row_is_flagged_and_routes_nothing():
    spec = O.LayerSpec(T=2, H=8, n_experts=4, n_sub=2, I_sub=4, k_max=4)
    Le = np.array([[1, 2, 3, 4], [4, 3, 2, 1]], dtype=np.float32)
    P = np.ones((2, 2, 2), dtype=np.float32)
    kappa = CG.default_kappa(4, 2, 2)
    kappa[3] = [2, 2]                            # sums to 4, not 3
    res = CG.route_cg(spec, None, None, None, None, 2, kappa, [3, 2], expert_logits=Le, proxy=P)
    assert res["flags"] & O.FLAG_K_RANGE
    assert (res["topk_idx"][0] == -1).all()
    assert (res["topk_idx"][1, :2] >= 0).all()


def test_package_allocation_table_equals_the_oracle_default():
    """The bench's input generator builds the allocation table on its own; it
    must equal the oracle's default rule on every workload shape."""
    from aware_moe_expert_gb300 import inputs as I, workloads as W
    for wl in W.ALL.values():
        got = I.allocation_table(wl.k_max, wl.native_m, wl.n_sub).numpy()
        np.testing.assert_array_equal(got, CG.default_kappa(wl.k_max, wl.native_m, wl.n_sub))
