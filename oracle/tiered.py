"""Plain CPU oracle of quality-tiered batching (host scheduling).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` call it.  It
shares no code with the library.

Source: "MoE-Prism: Model and System Support for Request-Level Compute
Elasticity in MoE Serving" (arXiv 2510.19366), §III-C2 "Temporal Separation
via Quality-Tiered Batching", Eq. (5).  Requests R_i = (a_i, n_i, k_i) wait in
a queue; a batch holds at most M prompt tokens and runs at one budget, the
largest of its requests.  The queue is sorted by (k, a); tiers are scanned in
ascending k and filled FIFO.  A tier that does not fill its last batch leaves a
residual of n_cur tokens at budget k; the next tier's leading requests that
still fit add n_next tokens, and the residual is promoted to k_next and merged
iff (n_cur + n_next) / T(n_cur + n_next, k_next) >= n_cur / T(n_cur, k);
otherwise it is dispatched at k.  T(n, k) is profiled at buckets and
interpolated.

Readings (where the page is silent):
  * "tokens contributed by the next tier under the remaining budget": that
    tier's requests taken in FIFO order while they fit, stopping at the first
    one that does not;
  * a promoted batch stays open: the tier's later requests keep filling it;
  * a request with more than M tokens forms a batch of its own;
  * equal (k, a) keep queue order;
  * interpolation: linear in n between buckets, end segments extended
    linearly (one bucket: proportional), linear in k between buckets, k
    clamped to the profiled range.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple


def _interp(xs: Sequence[int], ys: Sequence[float], x: float) -> float:
    if len(xs) == 1:
        return ys[0] * x / xs[0] if xs[0] != 0 else ys[0]
    i = 0
    while i + 2 < len(xs) and x > xs[i + 1]:
        i += 1
    f = (x - xs[i]) / (xs[i + 1] - xs[i])
    return ys[i] + f * (ys[i + 1] - ys[i])


def cost(n_points: Sequence[int], k_points: Sequence[int], t: Sequence[Sequence[float]],
         n: float, k: float) -> float:
    """T(n, k) from the profiled table t[k_index][n_index]."""
    kk = min(max(k, k_points[0]), k_points[-1])
    j = 0
    while j + 1 < len(k_points) and kk > k_points[j + 1]:
        j += 1
    y0 = _interp(n_points, t[j], n)
    if j + 1 >= len(k_points) or kk == k_points[j]:
        return y0
    y1 = _interp(n_points, t[j + 1], n)
    f = (kk - k_points[j]) / (k_points[j + 1] - k_points[j])
    return y0 + f * (y1 - y0)


def tier_schedule(reqs: Sequence[Tuple[float, int, int]], M: int, n_points, k_points, t
                  ) -> List[Tuple[int, List[int]]]:
    """Batches in dispatch order, each (budget, [request indices])."""
    T = lambda n, k: cost(n_points, k_points, t, n, k)  # noqa: E731
    order = sorted(range(len(reqs)), key=lambda i: (reqs[i][2], reqs[i][0], i))
    tiers: List[List[int]] = []
    for i in order:
        if tiers and reqs[tiers[-1][0]][2] == reqs[i][2]:
            tiers[-1].append(i)
        else:
            tiers.append([i])
    batches: List[Tuple[int, List[int]]] = []
    res = None          # open batch: [k, tokens, [requests]]
    for tier in tiers:
        k = reqs[tier[0]][2]
        rest = list(tier)
        if res is not None:
            n_cur = res[1]
            take, n_next = [], 0
            for i in rest:
                if n_cur + n_next + reqs[i][1] <= M:
                    take.append(i)
                    n_next += reqs[i][1]
                else:
                    break
            if take and (n_cur + n_next) / T(n_cur + n_next, k) >= n_cur / T(n_cur, res[0]):
                res = [k, n_cur + n_next, res[2] + take]
                rest = rest[len(take):]
            else:
                batches.append((res[0], res[2]))
                res = None
        for i in rest:
            if res is not None and res[1] + reqs[i][1] > M:
                batches.append((res[0], res[2]))
                res = None
            if res is None:
                res = [k, 0, []]
            res[1] += reqs[i][1]
            res[2].append(i)
    if res is not None:
        batches.append((res[0], res[2]))
    return batches
