"""Plain, slow fp64 CPU oracle for one k-aware Mixture-of-Experts layer forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU baseline
and its ``--impl reference`` arm) call it.  It shares no code with the CUDA
library and imports nothing from it.

What it computes is the exact definition of the layer, written out step by
step in float64 over the exact values of bf16-stored inputs:

  1. router logits   L[t,u] = x_t . router_w[u] + bias[u // n_sub]
  2. per-token top-k_t selection on L (ties to the lower unit index)
  3. gate weights    softmax over all units (or sigmoid), optional
                     renormalisation over the selected units, times route_scale
  4. permutation     assignments grouped by unit, ascending token inside a unit
  5. SwiGLU FFN      per assignment, no intermediate rounding
  6. combine         out_t = sum_j w_{t,j} * y_{t,j}  (+ shared expert, weight 1)

Sources (cited per function below):
  [Prism]  "MoE-Prism: Model and System Support for Request-Level Compute
           Elasticity in MoE Serving" (arXiv 2510.19366)
  [PCoMoE] "PCoMoE: Shifting MoE Inference from Monolithic Expert Selection to
           Fine-Grained Path Composition" (arXiv 2609.01024)

Readings taken where the pages are silent (each is also a test pin or noted):
  * selection is made on the logit (softmax and sigmoid are monotone); -0 and +0
    are equal, NaN sorts after every number, ties go to the lower unit index;
  * softmax runs over all E_r units; ``renorm`` divides by the selected sum;
  * the expert bias is added to the logit before both selection and gate and is
    shared by the n_sub sub-experts of an expert;
  * the shared expert is added with weight 1 and is not part of k.

Pinned: every function here is pinned by a test in tests/test_oracle_pins.py
against closed forms (one-hot weights reduce the layer to silu(x_a) x_b w at
output c), identities the pages state (all sub-experts of an expert at equal
gate equal the monolithic expert; k = E_r equals the dense gate-weighted sum;
the repeated-row router reproduces the unsplit layer) and brute force (top-k
against a full sort, the permutation enumerated on tiny inputs).  The pages
print no worked numerical example of a layer output, so there is no stored
value from them to compare against.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, Optional, Sequence

import numpy as np

SCORE_SOFTMAX = "softmax"
SCORE_SIGMOID = "sigmoid"

# Device-status style flags the oracle reports next to its results.
FLAG_NONFINITE = 1
FLAG_K_RANGE = 2


@dataclass
class LayerSpec:
    """Shape and routing options of one k-aware MoE layer.

    [Prism] §III-B1: an expert of intermediate size C = n_sub * I_sub is split
    into n_sub sub-experts of I_sub neurons each; unit u = e * n_sub + n.
    """
    T: int
    H: int
    n_experts: int
    n_sub: int
    I_sub: int
    k_max: int
    score: str = SCORE_SOFTMAX
    renorm: bool = False
    route_scale: float = 1.0
    I_shared: int = 0

    @property
    def E_r(self) -> int:
        return self.n_experts * self.n_sub


@dataclass
class FlopCounter:
    """Counts 2*m*n*k for every matrix product the oracle performs."""
    gate_up: int = 0
    down: int = 0
    router: int = 0
    shared: int = 0
    calls: list = field(default_factory=list)

    def add(self, kind: str, m: int, n: int, k: int) -> None:
        f = 2 * m * n * k
        setattr(self, kind, getattr(self, kind) + f)
        self.calls.append((kind, m, n, k))

    @property
    def routed(self) -> int:
        return self.gate_up + self.down


def bf16_to_f64(a) -> np.ndarray:
    """Exact float64 value of bf16 data.

    bf16 is the upper half of an IEEE binary32, so a uint16 bit pattern b has
    the value of the binary32 with bits (b << 16); binary32 -> binary64 is exact.
    Float arrays pass through (cast to float64, exact for float32/float64).
    """
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if a.dtype == np.int16:
        return bf16_to_f64(a.view(np.uint16))
    return a.astype(np.float64)


def _unit(w, u: int) -> np.ndarray:
    return bf16_to_f64(w(u) if callable(w) else w[u])


def router_logits(x, router_w, expert_bias, n_sub: int,
                  flops: Optional[FlopCounter] = None) -> np.ndarray:
    """L[t, u] = x_t . router_w[u] + bias[u // n_sub]   (float64, [T, E_r]).

    [Prism] §III-B2 "Low-Cost Fine-Tuning": the expanded linear gate is a plain
    linear layer scoring every sub-expert; the per-expert bias is broadcast to
    the n_sub sub-experts of that expert.
    """
    X = bf16_to_f64(x)
    R = bf16_to_f64(router_w)
    L = X @ R.T
    if flops is not None:
        flops.add("router", X.shape[0], R.shape[0], X.shape[1])
    if expert_bias is not None:
        b = np.asarray(expert_bias, dtype=np.float64)
        L = L + np.repeat(b, n_sub)[None, :]
    return L


def selection_order(logits_row: np.ndarray) -> np.ndarray:
    """Unit indices of one token ordered by (logit descending, index ascending).

    -0.0 and +0.0 compare equal; NaN sorts after every number (then by index).
    """
    L = np.asarray(logits_row, dtype=np.float64)
    nan = np.isnan(L)
    val = np.where(nan, 0.0, L) + 0.0          # + 0.0 turns -0.0 into +0.0
    idx = np.arange(L.shape[0])
    # lexsort: the last key is the primary one
    return np.lexsort((idx, -val, nan.astype(np.int8)))


def select_topk(logits: np.ndarray, k_per_token: Sequence[int], k_max: int):
    """Per-token top-k_t selection.  [Prism] §III-B2 (LG selects the top-k over
    all sub-experts) with the per-request budget k_i of §III-C1.

    Returns (topk_idx int32 [T, k_max] padded with -1, flags).  A k_t outside
    [1, k_max] sets FLAG_K_RANGE and is clamped into [0, k_max] so that the
    output stays well-formed; a non-finite logit sets FLAG_NONFINITE (infinite
    logits are still ordered, NaN last).
    """
    L = np.asarray(logits, dtype=np.float64)
    T, E_r = L.shape
    flags = 0
    if np.isnan(L).any() or np.isinf(L).any():
        flags |= FLAG_NONFINITE
    idx = np.full((T, k_max), -1, dtype=np.int32)
    for t in range(T):
        k = int(k_per_token[t])
        if k < 1 or k > k_max:
            flags |= FLAG_K_RANGE
            k = min(max(k, 0), k_max)
        k = min(k, E_r)
        idx[t, :k] = selection_order(L[t])[:k]
    return idx, flags


def gate_weights(logits: np.ndarray, topk_idx: np.ndarray, k_per_token,
                 score: str, renorm: bool, route_scale: float) -> np.ndarray:
    """Gate weight of every selected unit (float64 [T, k_max], 0 in padding).

    softmax: p_u = exp(L_u - max_v L_v) / sum_v exp(L_v - max_v L_v) over ALL
    units, w_j = p_{u_j}.  sigmoid: w_j = 1 / (1 + exp(-L_{u_j})).
    renorm divides by the sum over the k_t selected units; the result is then
    multiplied by route_scale ("retain the model's routing normalization and
    apply the N-adjusted routed scaling", [Prism] §III-B2).
    """
    L = np.asarray(logits, dtype=np.float64)
    T = L.shape[0]
    k_max = topk_idx.shape[1]
    w = np.zeros((T, k_max), dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        if score == SCORE_SOFTMAX:
            m = np.max(L, axis=1, keepdims=True)
            e = np.exp(L - m)
            s = e / np.sum(e, axis=1, keepdims=True)
        elif score == SCORE_SIGMOID:
            s = 1.0 / (1.0 + np.exp(-L))
        else:
            raise ValueError(score)
    for t in range(T):
        k = min(max(int(k_per_token[t]), 0), k_max)
        sel = topk_idx[t, :k]
        vals = s[t, sel]
        if renorm:
            vals = vals / np.sum(vals)
        w[t, :k] = vals * route_scale
    return w


def permute(topk_idx: np.ndarray, k_per_token, E_r: int):
    """Group the assignments (t, j) by routing unit.

    Order: unit ascending, token ascending inside a unit (each token selects a
    unit at most once, so this order is unique).  Returns counts [E_r],
    offsets [E_r + 1] (exclusive prefix sum), sorted_token [N_assign] and
    inv_row [T, k_max] (position of assignment (t, j), -1 in padding).
    [Prism] §II-D: grouped-GEMM kernels need the rows of one expert contiguous.
    """
    T, k_max = topk_idx.shape
    pairs = []
    for t in range(T):
        k = min(max(int(k_per_token[t]), 0), k_max)
        for j in range(k):
            pairs.append((int(topk_idx[t, j]), t, j))
    pairs.sort()
    counts = np.zeros(E_r, dtype=np.int32)
    for u, _, _ in pairs:
        counts[u] += 1
    offsets = np.zeros(E_r + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    sorted_token = np.array([t for _, t, _ in pairs], dtype=np.int32)
    inv_row = np.full((T, k_max), -1, dtype=np.int32)
    for pos, (_, t, j) in enumerate(pairs):
        inv_row[t, j] = pos
    return counts, offsets, sorted_token, inv_row


def silu(g: np.ndarray) -> np.ndarray:
    """SiLU(g) = g * sigmoid(g) = g / (1 + exp(-g))."""
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu_ffn(X: np.ndarray, w_gate_up_u: np.ndarray, w_down_u: np.ndarray,
               flops: Optional[FlopCounter] = None, kind: str = "routed") -> np.ndarray:
    """One (sub-)expert: A = SiLU(X Wg) * (X Wu), Y = A Wd.   [Prism] §III-B1 Eq. (1).

    Weight layout (out x in, as a linear layer): w_gate_up_u = [2I, H] with the
    gate neurons in rows 0..I-1 and the up neurons in rows I..2I-1; w_down_u =
    [H, I].  Everything in float64 with no intermediate rounding.
    """
    I = w_gate_up_u.shape[0] // 2
    Wg = w_gate_up_u[:I]
    Wu = w_gate_up_u[I:]
    G = X @ Wg.T
    U = X @ Wu.T
    A = silu(G) * U
    Y = A @ w_down_u.T
    if flops is not None:
        r, H = X.shape
        if kind == "routed":
            flops.add("gate_up", r, 2 * I, H)
            flops.add("down", r, H, I)
        else:
            flops.add("shared", r, 2 * I, H)
            flops.add("shared", r, H, I)
    return Y


def route(spec: LayerSpec, x=None, router_w=None, expert_bias=None,
          k_per_token=None, logits=None, flops: Optional[FlopCounter] = None):
    """Steps 1-3: logits (computed in float64 unless given), top-k_t, gates."""
    if logits is None:
        L = router_logits(x, router_w, expert_bias, spec.n_sub, flops)
    else:
        L = np.asarray(logits).astype(np.float64)
    idx, flags = select_topk(L, k_per_token, spec.k_max)
    w = gate_weights(L, idx, k_per_token, spec.score, spec.renorm, spec.route_scale)
    return L, idx, w, flags


def layer_forward(spec: LayerSpec, x, router_w, w_gate_up, w_down, k_per_token,
                  expert_bias=None, logits=None, w_shared_gate_up=None,
                  w_shared_down=None, routed=None) -> dict:
    """The whole layer forward, in the order of the method's steps.

    Output of token t ([Prism] §III-B2, the routed output sum_j w_j FFN_j(x)):
        out_t = sum_{j < k_t} w_{t,j} * FFN_{u_{t,j}}(x_t)  +  FFN_shared(x_t)
    Weights may be arrays indexed by unit or callables u -> array (bf16 bit
    patterns as uint16, or floats).  ``logits`` (float32 [T, E_r]) replaces
    step 1 when given; ``routed`` = (topk_idx, topk_w) replaces steps 1-3 (a
    routing made by another router, e.g. the proxy router).
    """
    flops = FlopCounter()
    X = bf16_to_f64(x)
    T, H = X.shape
    assert T == spec.T and H == spec.H
    if routed is None:
        L, idx, w, flags = route(spec, X, router_w, expert_bias, k_per_token, logits, flops)
    else:
        L, flags = None, 0
        idx = np.asarray(routed[0], dtype=np.int32)
        w = np.asarray(routed[1], dtype=np.float64)
    counts, offsets, sorted_token, inv_row = permute(idx, k_per_token, spec.E_r)
    n_assign = int(offsets[-1])
    y_perm = np.zeros((n_assign, H), dtype=np.float64)
    for u in range(spec.E_r):
        lo, hi = int(offsets[u]), int(offsets[u + 1])
        if hi == lo:
            continue
        rows = sorted_token[lo:hi]
        y_perm[lo:hi] = swiglu_ffn(X[rows], _unit(w_gate_up, u), _unit(w_down, u), flops)
    out = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        for j in range(spec.k_max):
            r = inv_row[t, j]
            if r >= 0:
                out[t] += w[t, j] * y_perm[r]
    y_shared = None
    if spec.I_shared > 0:
        y_shared = swiglu_ffn(X, bf16_to_f64(w_shared_gate_up), bf16_to_f64(w_shared_down),
                              flops, kind="shared")
        out += y_shared
    return dict(out=out, logits=L, topk_idx=idx, topk_w=w, counts=counts,
                offsets=offsets, sorted_token=sorted_token, inv_row=inv_row,
                y_perm=y_perm, y_shared=y_shared, flags=flags, flops=flops,
                n_assign=n_assign)


def layer_forward_routings(spec: LayerSpec, x, router_w, w_gate_up, w_down, k_per_token,
                           expert_bias=None, logits_list=(None,), w_shared_gate_up=None,
                           w_shared_down=None) -> list:
    """layer_forward for several routings of the same tokens at once.

    Each entry of ``logits_list`` fixes one routing: None routes on the
    float64 logits of step 1, an array routes on those logits (e.g. a GPU's
    fp32 logits).  Steps 2-3 run per routing; the SwiGLU FFN of every
    (token, unit) pair that any routing selects is evaluated once (no
    intermediate rounding) and each routing combines its own selection with
    its own gates, plus the shared expert with weight 1.  Returns one dict per
    routing: out, logits, topk_idx, topk_w, flags.
    """
    X = bf16_to_f64(x)
    T, H = X.shape
    assert T == spec.T and H == spec.H
    L64 = None
    routes = []
    for lg in logits_list:
        if lg is None:
            if L64 is None:
                L64 = router_logits(X, router_w, expert_bias, spec.n_sub)
            routes.append(route(spec, logits=L64, k_per_token=k_per_token))
        else:
            routes.append(route(spec, logits=lg, k_per_token=k_per_token))
    need = {}
    for _, idx, _, _ in routes:
        for t in range(T):
            for j in range(spec.k_max):
                u = int(idx[t, j])
                if u >= 0:
                    need.setdefault(u, set()).add(t)
    y = {}
    for u in sorted(need):
        rows = sorted(need[u])
        Y = swiglu_ffn(X[rows], _unit(w_gate_up, u), _unit(w_down, u))
        for r, t in enumerate(rows):
            y[(t, u)] = Y[r]
    y_shared = None
    if spec.I_shared > 0:
        y_shared = swiglu_ffn(X, bf16_to_f64(w_shared_gate_up), bf16_to_f64(w_shared_down))
    results = []
    for L, idx, w, flags in routes:
        out = np.zeros((T, H), dtype=np.float64)
        for t in range(T):
            for j in range(spec.k_max):
                u = int(idx[t, j])
                if u >= 0:
                    out[t] += w[t, j] * y[(t, u)]
        if y_shared is not None:
            out += y_shared
        results.append(dict(out=out, logits=L, topk_idx=idx, topk_w=w, flags=flags))
    return results


def coarse_k(k_qos: int, n_sub: int) -> int:
    """k_exec = N * ceil(k_qos / N): the budget a whole-expert layout must run
    to meet a target given in sub-expert units.  [Prism] §V-D1."""
    return n_sub * int(math.ceil(k_qos / n_sub))


def routed_flops(H: int, I_sub: int, k_per_token) -> int:
    """Algorithmic routed FLOPs: 6 * H * I_sub per assignment (gate and up:
    4*H*I_sub, two thirds, [PCoMoE] §3; down: 2*H*I_sub)."""
    return 6 * H * I_sub * int(np.sum(np.asarray(k_per_token, dtype=np.int64)))


def distinct_units(counts: np.ndarray) -> int:
    """D: number of routing units with at least one assignment."""
    return int(np.count_nonzero(np.asarray(counts)))
