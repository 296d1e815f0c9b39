"""Pins of the quality-tiered batching oracle (oracle/tiered.py), no GPU:
a hand-worked Eq. (5) example (tests/golden/tiered_batching.txt), the two
cost regimes whose answer is known in closed form, interpolation identities
and structural invariants on random queues."""
import os

import numpy as np
import pytest

from oracle import tiered as Q

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tiered_batching.txt")


def load_golden():
    n_points = k_points = None
    t, M, scen, cur = [], None, {}, None
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        f = line.split()
        if f[0] == "n_points":
            n_points = [int(v) for v in f[1:]]
        elif f[0] == "k_points":
            k_points = [int(v) for v in f[1:]]
        elif f[0] == "t":
            t.append([float(v) for v in f[2:]])
        elif f[0] == "M":
            M = int(f[1])
        elif f[0] == "scenario":
            cur = scen.setdefault(f[1], {"reqs": [], "batches": []})
        elif f[0] == "req":
            cur["reqs"].append((float(f[1]), int(f[2]), int(f[3])))
        elif f[0] == "batch":
            cur["batches"].append((int(f[1]), [int(v) for v in f[2:]]))
    return n_points, k_points, t, M, scen


@pytest.mark.parametrize("name", ["A", "B"])
def test_worked_example(name):
    n_points, k_points, t, M, scen = load_golden()
    got = Q.tier_schedule(scen[name]["reqs"], M, n_points, k_points, t)
    assert got == scen[name]["batches"]


def test_interpolation_identities():
    n_points, k_points, t = [100, 300, 700], [2, 6], [[10.0, 20.0, 60.0], [30.0, 50.0, 90.0]]
    for j, k in enumerate(k_points):
        for i, n in enumerate(n_points):
            assert Q.cost(n_points, k_points, t, n, k) == t[j][i]
    assert Q.cost(n_points, k_points, t, 200, 2) == pytest.approx(15.0)
    assert Q.cost(n_points, k_points, t, 100, 4) == pytest.approx(20.0)        # k midpoint
    assert Q.cost(n_points, k_points, t, 900, 2) == pytest.approx(80.0)        # extrapolated
    assert Q.cost(n_points, k_points, t, 50, 6) == pytest.approx(25.0)         # extrapolated
    assert Q.cost(n_points, k_points, t, 300, 1) == Q.cost(n_points, k_points, t, 300, 2)
    assert Q.cost(n_points, k_points, t, 300, 9) == Q.cost(n_points, k_points, t, 300, 6)
    assert Q.cost([400], [4], [[8.0]], 100, 4) == pytest.approx(2.0)           # proportional


def _queue(n, seed, ks=(2, 4, 6, 8)):
    rng = np.random.default_rng(seed)
    return [(float(rng.random()), int(rng.integers(32, 700)), int(rng.choice(ks)))
            for _ in range(n)]


def test_proportional_cost_never_promotes():
    """T(n, k) = c_k n with c_k increasing: n / T is 1/c_k, so promoting
    always lowers throughput; every batch holds one budget only."""
    reqs = _queue(60, 1)
    n_points, k_points = [64, 2048], [2, 4, 6, 8]
    t = [[c * 64, c * 2048] for c in (1.0, 2.0, 3.0, 4.0)]
    for k, b in Q.tier_schedule(reqs, 1024, n_points, k_points, t):
        assert {reqs[i][2] for i in b} == {k}


def test_constant_cost_always_promotes():
    """T(n, k) constant: more tokens always raise throughput, so a residual
    always merges with whatever of the next tier fits: every batch except
    the last is full up to the first request that does not fit."""
    reqs = _queue(60, 2)
    t = [[100.0, 100.0]] * 4
    out = Q.tier_schedule(reqs, 1024, [64, 2048], [2, 4, 6, 8], t)
    order = sorted(range(60), key=lambda i: (reqs[i][2], reqs[i][0], i))
    flat = [i for _, b in out for i in b]
    assert flat == order          # batches are consecutive runs of the sorted queue
    pos = 0
    for _, b in out[:-1]:
        pos += len(b)
        assert sum(reqs[i][1] for i in b) + reqs[order[pos]][1] > 1024


@pytest.mark.parametrize("seed", range(6))
def test_structural_invariants(seed):
    reqs = _queue(80, seed)
    reqs.append((0.5, 3000, 4))    # larger than M: a batch of its own
    n_points, k_points = [128, 512, 2048], [2, 4, 8]
    t = [[50 + k * n / 50 for n in n_points] for k in k_points]
    out = Q.tier_schedule(reqs, 1024, n_points, k_points, t)
    seen = sorted(i for _, b in out for i in b)
    assert seen == list(range(len(reqs)))
    for k, b in out:
        assert k == max(reqs[i][2] for i in b)
        tok = sum(reqs[i][1] for i in b)
        assert tok <= 1024 or len(b) == 1
    # FIFO inside a tier: dispatch order follows arrival
    pos = {i: p for p, i in enumerate(i for _, b in out for i in b)}
    for a in range(len(reqs)):
        for c in range(len(reqs)):
            if reqs[a][2] == reqs[c][2] and reqs[a][0] < reqs[c][0]:
                assert pos[a] < pos[c]
