"""The library's host scheduler (moe_tier_schedule, moe_cost_lookup in
libmoe.so, C++) against the oracle (oracle/tiered.py): identical batches on
the worked example and on random queues, identical interpolated costs, and
its argument checks.  Host code only: runs without a GPU."""
import numpy as np
import pytest

from aware_moe_expert_gb300 import binding as B
from oracle import tiered as Q
from test_oracle_tiered import load_golden


def _as_batches(batch_of, batch_k):
    out = [(k, []) for k in batch_k]
    for i, b in enumerate(batch_of):
        out[b][1].append(i)
    return out


def _dispatch_order(requests, batch_of):
    # the scheduler fills batches in dispatch order; inside a batch, members
    # appear in the order the oracle lists them (sorted queue order)
    order = sorted(range(len(requests)), key=lambda i: (requests[i][2], requests[i][0], i))
    out = {}
    for i in order:
        out.setdefault(batch_of[i], []).append(i)
    return [out[b] for b in sorted(out)]


@pytest.mark.parametrize("name", ["A", "B"])
def test_worked_example(name):
    n_points, k_points, t, M, scen = load_golden()
    table = B.CostTable(n_points, k_points, t)
    batch_of, bk, bt = B.moe_tier_schedule(scen[name]["reqs"], M, table)
    want = scen[name]["batches"]
    assert bk == [k for k, _ in want]
    assert _dispatch_order(scen[name]["reqs"], batch_of) == [b for _, b in want]
    assert bt == [sum(scen[name]["reqs"][i][1] for i in b) for _, b in want]


@pytest.mark.parametrize("seed", range(8))
def test_random_queues_match_oracle(seed):
    rng = np.random.default_rng(seed)
    reqs = [(float(rng.integers(0, 50)), int(rng.integers(16, 900)), int(rng.choice([2, 4, 6, 8])))
            for _ in range(int(rng.integers(1, 120)))]
    n_points = [128, 512, 2048, 8192]
    k_points = [2, 4, 6, 8]
    fixed = float(rng.uniform(0, 300))
    t = [[fixed + k * n * float(rng.uniform(0.005, 0.02)) for n in n_points] for k in k_points]
    for row in t:
        row.sort()
    M = int(rng.choice([512, 1024, 4096]))
    table = B.CostTable(n_points, k_points, t)
    batch_of, bk, _ = B.moe_tier_schedule(reqs, M, table)
    want = Q.tier_schedule(reqs, M, n_points, k_points, t)
    assert bk == [k for k, _ in want]
    assert _dispatch_order(reqs, batch_of) == [b for _, b in want]
    for n in (1, 100, 700, 5000, 20000):
        for k in (1, 2, 3, 5, 8, 9):
            assert B.moe_cost_lookup(table, n, k) == pytest.approx(
                Q.cost(n_points, k_points, t, n, k), rel=1e-12)


def test_rejects_bad_arguments():
    table = B.CostTable([128, 512], [2, 4], [[1.0, 2.0], [3.0, 4.0]])
    with pytest.raises(B.MoeError):
        B.moe_tier_schedule([(0.0, 0, 2)], 1024, table)          # empty request
    with pytest.raises(B.MoeError):
        B.moe_tier_schedule([(0.0, 10, 2)], 0, table)            # M < 1
    bad = B.CostTable([512, 128], [2, 4], [[1.0, 2.0], [3.0, 4.0]])
    with pytest.raises(B.MoeError):
        B.moe_tier_schedule([(0.0, 10, 2)], 1024, bad)           # buckets not increasing
    assert B.moe_cost_lookup(bad, 100, 2) == -1.0
    neg = B.CostTable([128, 512], [2, 4], [[1.0, -2.0], [3.0, 4.0]])
    assert B.moe_cost_lookup(neg, 100, 2) == -1.0                # times must be positive
