"""Plain fp64 CPU oracle of the training-free proxy router (CG) of a k-aware
MoE layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU baseline
and its ``--impl reference`` arm) call it.  It shares no code with the CUDA
library.

Source: "MoE-Prism: Model and System Support for Request-Level Compute
Elasticity in MoE Serving" (arXiv 2510.19366), §III-B2, "Gating Mechanism
Reconstructor" / "Training-Free Proxy Gating" (Fig. 7, left):

  offline   per expert, a calibration activation matrix A [B, C] gives a
            binary mask B[t, c] = 1 iff c is among the k_a largest |A[t, :]|;
            the co-activation matrix is C_co = B^T B; neuron i of sub-expert
            S_n scores sum_{j in S_n, j != i} C_co[i, j]; the r best form the
            gate-neuron set G_n.
  serving   the original router scores the original experts and keeps its
            native m of them, ordered by router probability, each with its
            normalised and scaled weight w_j.  For a selected expert j and each
            of its sub-experts n, the proxy score is
                s_n(x) = (1/r) sum_{c in G_n} |SiLU(x . Wg[c]) * (x . Wu[c])|.
            A configured allocation (kappa_1 .. kappa_m), 0 <= kappa_j <= N,
            sum_j kappa_j = k, keeps the kappa_j best sub-experts of expert j;
            each inherits w_j (no second softmax).  The routed output is
                sum_j w_j sum_{n in Top_kappa_j(s_j)} FFN_{j,n}(x).

Readings taken where the page is silent (also listed in the design notes):
  * "top kappa_j by proxy score": ties go to the lower sub-expert index; the
    expert-level selection uses the layer's own key (logit descending, lower
    index first, -0 == +0, NaN last) and its normalisation options;
  * the allocation for a per-token budget k_t is row k_t of a table
    kappa[k][j]; the default table splits k as evenly as possible, the
    higher-ranked experts taking the remainder;
  * the selected units of a token are listed expert by expert (router order),
    and inside an expert by proxy score (descending, lower index first);
  * k_a ties (equal |A| values) go to the lower neuron index, as do ties
    between gate-neuron scores;
  * neuron c of expert e belongs to sub-expert n = c // I_sub (the default
    contiguous partition), so gate neurons are stored as indices local to
    their sub-expert's rows.

Pinned by tests/test_oracle_cg_router.py: the full allocation reproduces the
unsplit top-m MoE, the proxy score has a closed form on one-hot weights, the
selection equals a brute-force sort, and the gate-neuron choice equals an
explicit pair count.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from . import moe_oracle as O


def topk_mask(A: np.ndarray, k_a: int) -> np.ndarray:
    """B[t, c] = 1 iff c is one of the k_a largest |A[t, :]| (ties: lower c)."""
    A = np.abs(np.asarray(A, dtype=np.float64))
    Bm = np.zeros(A.shape, dtype=np.int64)
    for t in range(A.shape[0]):
        order = np.lexsort((np.arange(A.shape[1]), -A[t]))
        Bm[t, order[:k_a]] = 1
    return Bm


def gate_neurons(A: np.ndarray, n_sub: int, k_a: int, r: int) -> np.ndarray:
    """Gate-neuron sets of one expert from its calibration activations.

    A [B, C] (C = n_sub * I_sub, contiguous partition).  Returns int32
    [n_sub, r]: for each sub-expert, the r local neuron indices (0..I_sub-1)
    with the largest co-activation with the other neurons of the same
    sub-expert, best first (ties: lower index).
    """
    Bm = topk_mask(A, k_a)
    Cco = Bm.T @ Bm                       # C_co = B^T B
    C = A.shape[1]
    I_sub = C // n_sub
    G = np.zeros((n_sub, r), dtype=np.int32)
    for n in range(n_sub):
        S = np.arange(n * I_sub, (n + 1) * I_sub)
        block = Cco[np.ix_(S, S)]
        score = block.sum(axis=1) - np.diag(block)     # exclude j == i
        order = np.lexsort((np.arange(I_sub), -score))
        G[n] = order[:r]
    return G


def default_kappa(k_max: int, m: int, n_sub: int) -> np.ndarray:
    """kappa[k][j] for k = 0..k_max: k split as evenly as possible over the m
    selected experts, the higher-ranked ones taking the remainder, each at
    most n_sub (requires k_max <= m * n_sub)."""
    assert k_max <= m * n_sub
    K = np.zeros((k_max + 1, m), dtype=np.int32)
    for k in range(k_max + 1):
        base, rem = divmod(k, m)
        K[k] = base + (np.arange(m) < rem)
    return K


def proxy_scores(x_row: np.ndarray, w_gate_up_units: Sequence[np.ndarray],
                 G_units: Sequence[np.ndarray]) -> np.ndarray:
    """s_n = (1/r) sum_{c in G_n} |SiLU(x . Wg_n[c]) * (x . Wu_n[c])| for the
    n_sub sub-experts of one expert.  w_gate_up_units[n] is the unit's
    [2 I_sub, H] block (gate rows, then up rows); G_units[n] its local gate
    neurons."""
    x = O.bf16_to_f64(x_row)
    s = np.zeros(len(w_gate_up_units), dtype=np.float64)
    for n, (W, G) in enumerate(zip(w_gate_up_units, G_units)):
        W = O.bf16_to_f64(W)
        I_sub = W.shape[0] // 2
        G = np.asarray(G, dtype=np.int64)
        g = W[G] @ x
        u = W[I_sub + G] @ x
        s[n] = np.mean(np.abs(O.silu(g) * u))
    return s


def sub_expert_order(scores: np.ndarray) -> np.ndarray:
    """Sub-experts of one expert ordered by proxy score descending, lower
    index first on ties (NaN after every number, as the layer's key)."""
    return O.selection_order(scores)


def route_cg(spec: O.LayerSpec, x, router_w_expert, w_gate_up, G, m: int, kappa,
             k_per_token, expert_bias=None, expert_logits=None, proxy=None) -> dict:
    """Training-free proxy routing of every token.

    spec describes the split layer (E_r = n_experts * n_sub units); its score,
    renorm and route_scale apply to the expert-level router.  G [E_r, r] holds
    each unit's local gate neurons; kappa [k_max + 1, m].  ``expert_logits``
    (float32 [T, n_experts]) and ``proxy`` (float32 [T, m, n_sub]) replace the
    oracle's own float64 values when given, so that a selection decided on
    another implementation's fp32 scores can be checked exactly.

    Returns expert_idx [T, m], expert_w [T, m], expert_logits, proxy [T, m,
    n_sub] (the values the selection used), topk_idx [T, k_max] (-1 padded),
    topk_w [T, k_max], flags.
    """
    N = spec.n_sub
    T = spec.T
    if expert_logits is None:
        Le = O.router_logits(x, router_w_expert, expert_bias, 1)
    else:
        Le = np.asarray(expert_logits).astype(np.float64)
    m_vec = np.full(T, m, dtype=np.int64)
    e_idx, flags = O.select_topk(Le, m_vec, m)
    e_w = O.gate_weights(Le, e_idx, m_vec, spec.score, spec.renorm, spec.route_scale)
    kappa = np.asarray(kappa, dtype=np.int64)
    X = O.bf16_to_f64(x) if proxy is None else None
    S = np.zeros((T, m, N), dtype=np.float64)
    topk_idx = np.full((T, spec.k_max), -1, dtype=np.int32)
    topk_w = np.zeros((T, spec.k_max), dtype=np.float64)
    for t in range(T):
        k = int(k_per_token[t])
        if k < 1 or k > spec.k_max:
            flags |= O.FLAG_K_RANGE
            k = min(max(k, 0), spec.k_max)
        row = kappa[k]
        if row.sum() != k or (row < 0).any() or (row > N).any():
            flags |= O.FLAG_K_RANGE
            continue
        slot = 0
        for j in range(m):
            e = int(e_idx[t, j])
            if proxy is None:
                units = [e * N + n for n in range(N)]
                S[t, j] = proxy_scores(X[t], [O._unit(w_gate_up, u) for u in units],
                                       [G[u] for u in units])
            else:
                S[t, j] = np.asarray(proxy[t, j], dtype=np.float64)
            order = sub_expert_order(S[t, j])
            for n in order[: int(row[j])]:
                topk_idx[t, slot] = e * N + int(n)
                topk_w[t, slot] = e_w[t, j]
                slot += 1
    return dict(expert_idx=e_idx, expert_w=e_w, expert_logits=Le, proxy=S,
                topk_idx=topk_idx, topk_w=topk_w, flags=flags)


def layer_forward_cg(spec: O.LayerSpec, x, router_w_expert, w_gate_up, w_down, G, m: int,
                     kappa, k_per_token, expert_bias=None, expert_logits=None,
                     proxy=None) -> dict:
    """The layer with the proxy router: sum_j w_j sum_{n in Top_kappa_j} FFN_{j,n}(x)."""
    r = route_cg(spec, x, router_w_expert, w_gate_up, G, m, kappa, k_per_token,
                 expert_bias, expert_logits, proxy)
    k_eff = np.asarray([int(np.sum(r["topk_idx"][t] >= 0)) for t in range(spec.T)])
    out = O.layer_forward(spec, x, None, w_gate_up, w_down, k_eff,
                          routed=(r["topk_idx"], r["topk_w"]))
    out["cg"] = r
    return out
