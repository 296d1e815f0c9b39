"""Plain CPU oracle of decode expert-pool folding (routing-metadata rewrite).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU baseline
and its ``--impl reference`` arm) call it.  It shares no code with the CUDA
library and imports nothing from it.

Source: "ExFold: Unified Expert Folding for Training-Free MoE Prefill-Decode
Acceleration" (arXiv 2608.24938), sections "Unified Expert Folding",
"Phase-Specific Selection and Unified Folding" and "Phase-Specific Routing and
Folding" (pp. 4, 12-13).  Decode cost follows the distinct experts a batch
activates; ExFold bounds that set to a pool of D experts and folds every route
to an expert outside the pool into a retained target: the excluded
contribution alpha_e E_e(x) is approximated by alpha_e S[e, tau] E_tau(x), the
target tau being the pool member with the smallest calibrated projection loss
L[e, tau], so the scalar only changes the target's router weight.  Routes of a
token that land on the same target are coalesced, so each retained target runs
once per token.  The pool is either dynamic (ranked by the batch's aggregate
routed contribution) or static (fixed in advance).

What it computes (the plainest reading; every choice is also a test pin or a
listed reading), all in float64 over the fp32 inputs (routed weights, S, h):

  1. pool (dynamic): score_u = h_u * sum of the routed weights of unit u over
     the batch (exact real-number definition, evaluated in float64); the D
     best units by score (larger first, lower index on ties) form the pool;
     units nobody routes to (score 0 is never positive) join only if fewer
     than D units carry weight, again by lower index.
  2. target map: tau(u) = u for a pool member; otherwise the pool member p with
     the smallest L[u, p] (lower index on ties, a NaN loss counting as +inf),
     with scale S[u, tau(u)].
  3. remap: route (t, j) of unit u and weight w becomes (tau(u), w * S[u, tau])
     (float64 product); a pool member keeps its weight unchanged.
  4. coalesce: per token, routes with the same target are merged (their
     weights added) at the position of their first occurrence; the token's
     new budget is the number of distinct targets.

A GPU evaluates the sums of steps 1 and 4 in fp32 in some order; the
difference from the float64 value is bounded by ``score_error_bound`` (and,
for a merged weight, the same bound over its terms), so a pool member that
differs from the oracle's must lie within that bound of the selection
boundary (a near tie), and merged weights agree within it.

Readings (where the page is silent): the pages' experts are this layer's
routing units (sub-experts when the experts are split); the per-unit
magnitude h (the page ranks by router score times output magnitude) defaults
to 1; S and L are calibration tables the caller supplies (synthetic here:
calibration data are out of scope).
"""
from __future__ import annotations

from typing import Optional

import numpy as np

U32 = 2.0 ** -24     # unit roundoff of fp32


def gamma(n: int) -> float:
    """gamma_n = n u / (1 - n u): the relative error bound of n fp32 roundings
    (Higham, "Accuracy and Stability of Numerical Algorithms", Lemma 3.1)."""
    return n * U32 / (1.0 - n * U32)


def pool_scores(topk_idx: np.ndarray, topk_w: np.ndarray, k_per_token, E_r: int,
                unit_scale: Optional[np.ndarray] = None) -> np.ndarray:
    """Step 1's score: h_u times the aggregate routed weight of unit u, in
    float64 (the weights are fp32 numbers, exact in float64)."""
    T = topk_idx.shape[0]
    total = np.zeros(E_r, dtype=np.float64)
    for t in range(T):
        for j in range(int(k_per_token[t])):
            total[int(topk_idx[t, j])] += float(np.float32(topk_w[t, j]))
    if unit_scale is not None:
        total = total * np.asarray(unit_scale, dtype=np.float32).astype(np.float64)
    return total


def score_error_bound(topk_idx: np.ndarray, topk_w: np.ndarray, k_per_token, E_r: int,
                      unit_scale: Optional[np.ndarray] = None) -> np.ndarray:
    """Per unit, a bound on |fp32 evaluation - score_u| for ANY order of the
    fp32 additions followed by one fp32 product with h_u: a sum of n terms
    rounds n - 1 times, the product once, so the error is at most
    gamma_n * |h_u| * sum |w| (n = the unit's route count)."""
    T = topk_idx.shape[0]
    abs_sum = np.zeros(E_r, dtype=np.float64)
    n = np.zeros(E_r, dtype=np.int64)
    for t in range(T):
        for j in range(int(k_per_token[t])):
            u = int(topk_idx[t, j])
            abs_sum[u] += abs(float(np.float32(topk_w[t, j])))
            n[u] += 1
    h = np.ones(E_r) if unit_scale is None else \
        np.abs(np.asarray(unit_scale, dtype=np.float32).astype(np.float64))
    return np.array([gamma(int(n[u]) + 1) for u in range(E_r)]) * h * abs_sum


def select_pool(scores: np.ndarray, D: int) -> np.ndarray:
    """The D best units: score descending, lower index first on ties
    (-0 equals +0; a NaN score ranks below every number)."""
    E_r = scores.shape[0]
    s = np.asarray(scores, dtype=np.float64)
    key = np.where(np.isnan(s), -np.inf, s)
    key = np.where(key == 0.0, 0.0, key)
    order = sorted(range(E_r), key=lambda u: (-key[u], u))
    return np.array(sorted(order[:min(D, E_r)]), dtype=np.int64)


def target_map(pool: np.ndarray, S: np.ndarray, L: np.ndarray, E_r: int):
    """tau(u) and its scale: a pool member maps to itself with scale 1,
    any other unit to the pool member of least L[u, p] (lower p on ties; a
    NaN loss counts as +inf)."""
    in_pool = np.zeros(E_r, dtype=bool)
    in_pool[pool] = True
    tau = np.empty(E_r, dtype=np.int64)
    scale = np.empty(E_r, dtype=np.float32)
    for u in range(E_r):
        if in_pool[u]:
            tau[u], scale[u] = u, np.float32(1.0)
            continue
        def loss(p):
            v = float(L[u, p])
            return np.inf if np.isnan(v) else v
        best = None
        for p in sorted(int(v) for v in pool):
            if best is None or loss(p) < loss(best):
                best = p
        tau[u] = best
        scale[u] = np.float32(S[u, best])
    return tau, scale


def fold_routes(topk_idx: np.ndarray, topk_w: np.ndarray, k_per_token, tau: np.ndarray,
                scale: np.ndarray, in_pool: np.ndarray, return_abs: bool = False):
    """Steps 3-4: remap every route to its target and coalesce per token, in
    float64.

    Returns (idx [T, k_max] with -1 after the new budget, w [T, k_max] float64
    with 0 there, k_new [T]); with return_abs also (abs_terms [T, k_max]: the
    sum of |term| and the number of terms merged into every entry, for the
    rounding bound of an fp32 evaluation)."""
    T, k_max = topk_idx.shape
    idx_out = np.full((T, k_max), -1, dtype=np.int64)
    w_out = np.zeros((T, k_max), dtype=np.float64)
    abs_out = np.zeros((T, k_max), dtype=np.float64)
    n_out = np.zeros((T, k_max), dtype=np.int64)
    k_out = np.zeros(T, dtype=np.int64)
    for t in range(T):
        targets, weights, mags, terms = [], [], [], []
        for j in range(int(k_per_token[t])):
            u = int(topk_idx[t, j])
            w = float(np.float32(topk_w[t, j]))
            if not in_pool[u]:
                w = w * float(np.float32(scale[u]))
            v = int(tau[u])
            if v in targets:
                i = targets.index(v)
                weights[i] += w
                mags[i] += abs(w)
                terms[i] += 1
            else:
                targets.append(v)
                weights.append(w)
                mags.append(abs(w))
                terms.append(1)
        k_out[t] = len(targets)
        idx_out[t, :len(targets)] = targets
        w_out[t, :len(targets)] = weights
        abs_out[t, :len(targets)] = mags
        n_out[t, :len(targets)] = terms
    if return_abs:
        return idx_out, w_out, k_out, (abs_out, n_out)
    return idx_out, w_out, k_out


def fold_decode(topk_idx: np.ndarray, topk_w: np.ndarray, k_per_token, E_r: int, D: int,
                S: np.ndarray, L: np.ndarray, pool: Optional[np.ndarray] = None,
                unit_scale: Optional[np.ndarray] = None, return_abs: bool = False):
    """The whole rewrite: (idx, w, k_new, pool) (+ the merged terms' magnitudes
    with return_abs, see fold_routes).  pool=None: dynamic pool of D."""
    if pool is None:
        pool = select_pool(pool_scores(topk_idx, topk_w, k_per_token, E_r, unit_scale), D)
    pool = np.array(sorted(int(p) for p in pool), dtype=np.int64)
    in_pool = np.zeros(E_r, dtype=bool)
    in_pool[pool] = True
    tau, scale = target_map(pool, S, L, E_r)
    if return_abs:
        idx, w, k, mags = fold_routes(topk_idx, topk_w, k_per_token, tau, scale, in_pool, True)
        return idx, w, k, pool, mags
    idx, w, k = fold_routes(topk_idx, topk_w, k_per_token, tau, scale, in_pool)
    return idx, w, k, pool
