"""Pins of the decode expert-pool folding oracle (oracle/exfold.py), no GPU.

Each pin checks the oracle against something other than itself: a worked
example (tests/golden/exfold_fold.txt), the no-op case, the layer algebra the
fold stands for (computed by a separate uncoalesced loop), and brute-force
invariants of the pool and target choices.
"""
import os

import numpy as np
import pytest

from oracle import exfold as F
from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "exfold_fold.txt")


def _load_golden():
    E_r = D = k_max = None
    routes, L, S, pool, expect = {}, [], [], None, {}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        f = line.split()
        if f[0] == "E_r":
            E_r = int(f[1])
        elif f[0] == "D":
            D = int(f[1])
        elif f[0] == "k_max":
            k_max = int(f[1])
        elif f[0] in ("route", "expect"):
            pairs = [(int(a), float(b)) for a, b in (p.split(":") for p in f[2:])]
            (routes if f[0] == "route" else expect)[int(f[1])] = pairs
        elif f[0] == "L":
            L.append((int(f[1]), int(f[2]), float(f[3])))
        elif f[0] == "S":
            S.append((int(f[1]), int(f[2]), float(f[3])))
        elif f[0] == "pool":
            pool = [int(v) for v in f[1:]]
    T = len(routes)
    idx = np.full((T, k_max), -1, dtype=np.int64)
    w = np.zeros((T, k_max), dtype=np.float32)
    k = np.zeros(T, dtype=np.int64)
    for t, pairs in routes.items():
        k[t] = len(pairs)
        for j, (u, wt) in enumerate(pairs):
            idx[t, j], w[t, j] = u, wt
    Lm = np.full((E_r, E_r), 9.0, dtype=np.float32)
    Sm = np.ones((E_r, E_r), dtype=np.float32)
    for a, b, v in L:
        Lm[a, b] = v
    for a, b, v in S:
        Sm[a, b] = v
    return E_r, D, idx, w, k, Lm, Sm, pool, expect


def test_worked_example():
    """Pool (with an fp32 score tie), loss ties, scaled and coalesced routes
    as worked by hand in the fixture."""
    E_r, D, idx, w, k, L, S, pool, expect = _load_golden()
    oi, ow, ok, op = F.fold_decode(idx, w, k, E_r, D, S, L)
    assert op.tolist() == pool
    for t, pairs in expect.items():
        assert ok[t] == len(pairs)
        assert oi[t, :ok[t]].tolist() == [u for u, _ in pairs]
        np.testing.assert_allclose(ow[t, :ok[t]], [v for _, v in pairs], rtol=1e-6, atol=1e-7)
        assert (oi[t, ok[t]:] == -1).all() and (ow[t, ok[t]:] == 0).all()


def _random_routing(T, E_r, k_max, seed):
    rng = np.random.default_rng(seed)
    k = rng.integers(1, k_max + 1, T)
    idx = np.full((T, k_max), -1, dtype=np.int64)
    w = np.zeros((T, k_max), dtype=np.float32)
    for t in range(T):
        idx[t, :k[t]] = rng.choice(E_r, k[t], replace=False)
        w[t, :k[t]] = rng.random(k[t]).astype(np.float32)
    return idx, w, k


def _tables(E_r, seed):
    rng = np.random.default_rng(seed)
    S = np.clip(rng.normal(1.0, 0.5, (E_r, E_r)), -4, 4).astype(np.float32)
    np.fill_diagonal(S, 1.0)
    L = rng.random((E_r, E_r)).astype(np.float32)
    np.fill_diagonal(L, 0.0)
    return S, L


def test_pool_covering_every_routed_unit_is_a_no_op():
    """D at least the number of routed units: nothing is excluded, so the
    routing comes back unchanged (routes of one token are distinct units)."""
    idx, w, k = _random_routing(40, 24, 6, 1)
    S, L = _tables(24, 2)
    used = len(set(idx[idx >= 0].tolist()))
    oi, ow, ok, pool = F.fold_decode(idx, w, k, 24, used, S, L)
    np.testing.assert_array_equal(ok, k)
    np.testing.assert_array_equal(oi, idx)
    np.testing.assert_array_equal(ow, w)


@pytest.mark.parametrize("D", [1, 3, 8])
def test_folded_layer_equals_uncoalesced_sum(D):
    """The folded routing computes out_t = sum over the ORIGINAL routes of
    w * S[u, tau(u)] * FFN_tau(u)(x_t) (weight 1 scale for pool members): a
    separate loop over the original routes, without coalescing, in fp64."""
    rng = np.random.default_rng(7)
    T, H, E_r, I_sub, k_max = 12, 16, 10, 8, 4
    idx, w, k = _random_routing(T, E_r, k_max, 3)
    S, L = _tables(E_r, 4)
    x = rng.normal(size=(T, H))
    wgu = rng.normal(size=(E_r, 2 * I_sub, H)) / 4
    wd = rng.normal(size=(E_r, H, I_sub)) / 4
    oi, ow, ok, pool = F.fold_decode(idx, w, k, E_r, D, S, L)
    got = np.zeros((T, H))
    for t in range(T):
        for j in range(ok[t]):
            u = oi[t, j]
            got[t] += float(ow[t, j]) * O.swiglu_ffn(x[t:t + 1], wgu[u], wd[u])[0]
    in_pool = set(pool.tolist())
    want = np.zeros((T, H))
    for t in range(T):
        for j in range(k[t]):
            u = idx[t, j]
            if u in in_pool:
                tgt, sc = u, 1.0
            else:
                tgt = min(pool, key=lambda p: (L[u, p], p))
                sc = float(S[u, tgt])
            want[t] += float(np.float32(np.float32(w[t, j]) * np.float32(sc))) * \
                O.swiglu_ffn(x[t:t + 1], wgu[tgt], wd[tgt])[0]
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-6)


def test_pool_and_targets_satisfy_their_definitions():
    """Brute-force invariants: every pool score >= every other score, ties to
    the lower index; every target is the least-loss pool member (lower index on
    ties); after folding every target is in the pool and a token's targets are
    distinct."""
    for seed in range(5):
        idx, w, k = _random_routing(70, 32, 8, seed)
        S, L = _tables(32, seed + 10)
        L[np.random.default_rng(seed).random(L.shape) < 0.2] = 0.5   # loss ties
        D = 5
        sc = F.pool_scores(idx, w, k, 32)
        oi, ow, ok, pool = F.fold_decode(idx, w, k, 32, D, S, L)
        inside = set(pool.tolist())
        assert len(inside) == D
        for u in inside:
            for v in set(range(32)) - inside:
                assert sc[u] > sc[v] or (sc[u] == sc[v] and u < v)
        tau, _ = F.target_map(pool, S, L, 32)
        for u in set(range(32)) - inside:
            for p in inside:
                assert L[u, tau[u]] < L[u, p] or (L[u, tau[u]] == L[u, p] and tau[u] <= p)
        for t in range(70):
            tg = oi[t, :ok[t]].tolist()
            assert set(tg) <= inside and len(tg) == len(set(tg))


def test_pool_scores_are_the_exact_aggregate_weight():
    """The score is the real-number sum of each unit's fp32 routed weights
    (times h): math.fsum (correctly rounded) agrees to float64 rounding, and
    a separate per-route loop with h applied route by route gives the same."""
    import math
    idx, w, k = _random_routing(200, 16, 6, 5)
    h = np.random.default_rng(6).random(16).astype(np.float32) + 0.5
    got = F.pool_scores(idx, w, k, 16, unit_scale=h)
    terms = [[] for _ in range(16)]
    for t in range(200):
        for j in range(k[t]):
            terms[idx[t, j]].append(float(w[t, j]) * float(h[idx[t, j]]))
    want = np.array([math.fsum(v) for v in terms])
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=0)


def test_fp32_evaluations_stay_within_the_stated_bound():
    """Any fp32 order of the score's additions (forward, reversed, in
    64-token blocks) then the fp32 product with h lands within
    score_error_bound of the exact score."""
    idx, w, k = _random_routing(300, 24, 8, 8)
    h = np.random.default_rng(9).random(24).astype(np.float32) + 0.5
    exact = F.pool_scores(idx, w, k, 24, unit_scale=h)
    bound = F.score_error_bound(idx, w, k, 24, unit_scale=h)
    seqs = [[] for _ in range(24)]
    for t in range(300):
        for j in range(k[t]):
            seqs[idx[t, j]].append(np.float32(w[t, j]))
    for order in ("forward", "reverse", "blocks"):
        for u in range(24):
            v = seqs[u] if order != "reverse" else seqs[u][::-1]
            if order == "blocks":
                acc = np.float32(0)
                for b0 in range(0, len(v), 7):
                    part = np.float32(0)
                    for x in v[b0:b0 + 7]:
                        part = np.float32(part + x)
                    acc = np.float32(acc + part)
            else:
                acc = np.float32(0)
                for x in v:
                    acc = np.float32(acc + x)
            ev = float(np.float32(acc * h[u]))
            assert abs(ev - exact[u]) <= bound[u], (order, u)


def test_worked_example_tells_the_exact_score_from_an_fp32_sum():
    """Mutation check on the fixture: with the score added in fp32 (any
    order; the fixture's unit has two terms) the pool would be {0, 1}, not
    the exact sum's {1, 5}; the fixture therefore fails an oracle that
    evaluates the score in fp32."""
    E_r, D, idx, w, k, L, S, pool, expect = _load_golden()
    fp32 = np.zeros(E_r, dtype=np.float32)
    for t in range(idx.shape[0]):
        for j in range(k[t]):
            fp32[idx[t, j]] = np.float32(fp32[idx[t, j]] + w[t, j])
    assert F.select_pool(fp32, D).tolist() == [0, 1]
    assert F.select_pool(F.pool_scores(idx, w, k, E_r), D).tolist() == pool == [1, 5]


def test_exact_score_tie_goes_to_the_lower_index():
    """0.25 + 0.5 and 0.75 are exact in any precision: a true tie, the lower
    unit index enters the pool."""
    idx = np.array([[3, 1], [3, -1]])
    w = np.array([[0.75, 0.25], [0.0, 0.0]], dtype=np.float32)
    idx2 = np.array([[4, 1], [1, -1]])
    w2 = np.array([[0.75, 0.25], [0.5, 0.0]], dtype=np.float32)
    # unit 1: 0.25 + 0.5 = 0.75, unit 4: 0.75
    assert F.select_pool(F.pool_scores(idx2, w2, [2, 1], 6), 1).tolist() == [1]
    sc = F.pool_scores(idx, w, [2, 1], 6)
    assert sc[3] == 0.75 and sc[1] == 0.25


def test_static_pool_and_unit_scale():
    """A caller-given pool is used as is; a unit scale reorders the dynamic
    pool (score = scale * routed weight)."""
    idx, w, k = _random_routing(30, 12, 4, 9)
    S, L = _tables(12, 11)
    oi, ow, ok, pool = F.fold_decode(idx, w, k, 12, 3, S, L, pool=np.array([7, 2, 11]))
    assert pool.tolist() == [2, 7, 11]
    assert set(oi[oi >= 0].tolist()) <= {2, 7, 11}
    h = np.zeros(12, dtype=np.float32)
    h[[0, 5, 9]] = 1.0
    _, _, _, pool2 = F.fold_decode(idx, w, k, 12, 3, S, L, unit_scale=h)
    routed = F.pool_scores(idx, w, k, 12)
    if (routed[[0, 5, 9]] > 0).all():
        assert pool2.tolist() == [0, 5, 9]


def test_nan_loss_is_never_preferred():
    """A NaN projection loss counts as +inf: the finite least loss wins even
    when the NaN belongs to the lowest-index pool member; all-NaN falls back
    to the lowest index."""
    E_r = 5
    L = np.ones((E_r, E_r), dtype=np.float32)
    S = np.ones((E_r, E_r), dtype=np.float32)
    L[3, 0], L[3, 1], L[3, 2] = np.nan, 0.7, 0.4
    L[4, :3] = np.nan
    tau, _ = F.target_map(np.array([0, 1, 2]), S, L, E_r)
    assert tau[3] == 2 and tau[4] == 0
