"""Plain fp64 CPU oracle of path-composed MoE execution with source-grouped
reuse.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` call it.  It
shares no code with the CUDA library.

Source: "PCoMoE: Shifting MoE Inference from Monolithic Expert Selection to
Fine-Grained Path Composition" (arXiv 2609.01024), sections on the
expansion-projection decomposition, the compositional path P_{i,j} and
"Source-Grouped Compute Reuse" (Figure 8).  A SwiGLU expert e splits into an
expansion side U_e(h) = SiLU(h W_gate_e) * (h W_up_e) and a projection side
D_e(z) = z W_down_e, so F_e = D_e(U_e(h)).  A path (i, j) composes the
expansion of source i with the projection of target j: P_{i,j}(h) =
D_j(U_i(h)).  A token with active paths Pi(h) and weights beta_{i,j} gives
    y(h) = sum_{(i,j) in Pi(h)} beta_{i,j} D_j(U_i(h)),
and source-grouped execution evaluates each U_i once per unique source:
    y(h) = sum_{i in S(h)} sum_{j in T_i(h)} beta_{i,j} D_j(U_i(h)).
Diagonal paths (i, i) with beta = alpha_i are the vanilla MoE layer.

The page's equations are missing from the extracted text; the formulas above
are the ones its prose defines (expansion = gate and up with the SiLU
product, projection = down, path = ordered composition, output = weighted
sum over active paths).  Path selection (a compatibility bias learned by
fine-tuning) is out of scope: paths arrive as inputs.

Readings: the page's experts are this layer's routing units; a token's
sources are listed in first-occurrence order of its paths; several paths of
a token may share a target (and a source); the shared expert, when given,
adds with weight 1; everything is fp64 with no intermediate rounding.

Pinned (tests/test_oracle_pcomoe.py): diagonal paths = the vanilla layer;
source grouping = per-path recomputation; one-hot closed forms for the
source/target roles, for paths sharing a target and for the shared-expert
term; unique-source bookkeeping by brute force.
"""
from __future__ import annotations

from typing import Callable, Sequence

import numpy as np


def silu(g: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def expansion(h: np.ndarray, w_gate_up_u: np.ndarray) -> np.ndarray:
    """U(h) = SiLU(h Wg^T) * (h Wu^T), w_gate_up_u = [2I, H] (gate rows first)."""
    I = w_gate_up_u.shape[0] // 2
    return silu(h @ w_gate_up_u[:I].T) * (h @ w_gate_up_u[I:].T)


def projection(z: np.ndarray, w_down_u: np.ndarray) -> np.ndarray:
    """D(z) = z Wd^T, w_down_u = [H, I]."""
    return z @ w_down_u.T


def unique_sources(src_idx: np.ndarray, n_paths: Sequence[int]):
    """Per token: the distinct sources in first-occurrence order and, for
    every path, the position of its source in that list."""
    T, k_max = src_idx.shape
    srcs = np.full((T, k_max), -1, dtype=np.int64)
    n_src = np.zeros(T, dtype=np.int64)
    slot = np.full((T, k_max), -1, dtype=np.int64)
    for t in range(T):
        seen: list = []
        for j in range(int(n_paths[t])):
            s = int(src_idx[t, j])
            if s not in seen:
                seen.append(s)
            slot[t, j] = seen.index(s)
        n_src[t] = len(seen)
        srcs[t, :len(seen)] = seen
    return srcs, n_src, slot


def paths_forward(x: np.ndarray, w_gate_up: Callable[[int], np.ndarray],
                  w_down: Callable[[int], np.ndarray], src_idx: np.ndarray,
                  tgt_idx: np.ndarray, beta: np.ndarray, n_paths: Sequence[int],
                  w_shared_gate_up=None, w_shared_down=None):
    """Source-grouped execution: one expansion per (token, unique source),
    one projection per path, plus a shared expert with weight 1 when given.
    Returns (out [T, H], expansions evaluated)."""
    T = x.shape[0]
    srcs, n_src, slot = unique_sources(src_idx, n_paths)
    out = np.zeros((T, x.shape[1]))      # the projection maps back to H
    n_exp = 0
    for t in range(T):
        z = [expansion(x[t:t + 1], w_gate_up(int(srcs[t, s]))) for s in range(int(n_src[t]))]
        n_exp += len(z)
        for j in range(int(n_paths[t])):
            out[t] += float(beta[t, j]) * projection(z[int(slot[t, j])],
                                                     w_down(int(tgt_idx[t, j])))[0]
    if w_shared_gate_up is not None:
        out += projection(expansion(x, w_shared_gate_up), w_shared_down)
    return out, n_exp
