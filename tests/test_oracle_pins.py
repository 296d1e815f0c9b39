"""Pins of the fp64 oracle against what the pages and mathematics fix.

Every check here ties the oracle to something other than itself: closed forms
(golden fixtures), brute force on tiny inputs, an independent per-neuron
formulation of the expert (MoE-Prism §III-B1 Eq. (2)), a library softmax, or a
structural identity stated on the pages (sub-expert split, repeated-row linear
gate, coarse execution budget).  No GPU is needed.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# Independent, deliberately naive formulations used only by the pins.
# ----------------------------------------------------------------------------

def _sig(z):
    return 1.0 / (1.0 + math.exp(-z)) if z > -700 else 0.0


def neuron_sum_expert(x, Wg, Wu, Wd):
    """MoE-Prism §III-B1 Eq. (2): X'_q = sum_d A_d * Wdown[d, q], one neuron at a
    time, with A_d = SiLU(x . Wg[d]) * (x . Wu[d]).  Wg, Wu: [I, H]; Wd: [H, I]."""
    H = len(x)
    y = [0.0] * Wd.shape[0]
    for d in range(Wg.shape[0]):
        g = float(np.dot(x, Wg[d]))
        v = float(np.dot(x, Wu[d]))
        a = g * _sig(g) * v
        for q in range(Wd.shape[0]):
            y[q] += a * Wd[q, d]
    return np.array(y)


def naive_moe(x, router_w, Wg, Wu, Wd, k, score="softmax", renorm=False, scale=1.0, bias=None):
    """Plain per-token MoE with whole experts given as lists of (Wg, Wu, Wd)."""
    T = x.shape[0]
    E = router_w.shape[0]
    logits = [[float(np.dot(x[t], router_w[e])) + (0.0 if bias is None else bias[e])
               for e in range(E)] for t in range(T)]
    return naive_moe_from_logits(x, logits, Wg, Wu, Wd, k, score, renorm, scale)


def naive_moe_from_logits(x, logits, Wg, Wu, Wd, k, score="softmax", renorm=False, scale=1.0):
    """naive_moe on given router logits [T][E]."""
    T = x.shape[0]
    out = np.zeros((T, Wd[0].shape[0]))
    for t in range(T):
        logit = [float(v) for v in logits[t]]
        E = len(logit)
        # brute-force top-k: repeatedly take the largest, lower index on ties
        left = list(range(E))
        sel = []
        for _ in range(k[t]):
            best = left[0]
            for e in left[1:]:
                if logit[e] > logit[best]:
                    best = e
            sel.append(best)
            left.remove(best)
        if score == "softmax":
            m = max(logit)
            z = sum(math.exp(l - m) for l in logit)
            s = {e: math.exp(logit[e] - m) / z for e in sel}
        else:
            s = {e: _sig(logit[e]) for e in sel}
        tot = sum(s.values())
        for e in sel:
            w = (s[e] / tot if renorm else s[e]) * scale
            out[t] += w * neuron_sum_expert(x[t], Wg[e], Wu[e], Wd[e])
    return out


def split_experts(Wg, Wu, Wd, n_sub, parts=None):
    """Slice monolithic experts into n_sub sub-experts along the neuron axis
    (MoE-Prism §III-B1 Eq. (3)); ``parts[e]`` is a permutation of the neurons
    (contiguous partition when None).  Returns (w_gate_up [E*n_sub, 2I_sub, H],
    w_down [E*n_sub, H, I_sub])."""
    E, I, H = Wg.shape
    I_sub = I // n_sub
    wgu = np.zeros((E * n_sub, 2 * I_sub, H))
    wd = np.zeros((E * n_sub, H, I_sub))
    for e in range(E):
        perm = np.arange(I) if parts is None else parts[e]
        for n in range(n_sub):
            S = perm[n * I_sub:(n + 1) * I_sub]
            u = e * n_sub + n
            wgu[u, :I_sub] = Wg[e][S]
            wgu[u, I_sub:] = Wu[e][S]
            wd[u] = Wd[e][:, S]
    return wgu, wd


def rel_err(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ----------------------------------------------------------------------------
# P1  all sub-experts with an equal gate == the monolithic expert
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("n_sub", [1, 2, 3, 4])
@pytest.mark.parametrize("random_partition", [False, True])
def test_p1_subexperts_reconstruct_expert(n_sub, random_partition):
    rng = np.random.default_rng(10 + n_sub)
    T, H, I = 5, 16, 24
    Wg = rng.normal(size=(1, I, H)) / math.sqrt(H)
    Wu = rng.normal(size=(1, I, H)) / math.sqrt(H)
    Wd = rng.normal(size=(1, H, I)) / math.sqrt(I)
    x = rng.normal(size=(T, H))
    parts = [rng.permutation(I)] if random_partition else None
    wgu, wd = split_experts(Wg, Wu, Wd, n_sub, parts)
    spec = O.LayerSpec(T=T, H=H, n_experts=1, n_sub=n_sub, I_sub=I // n_sub, k_max=n_sub,
                       score="softmax", renorm=False, route_scale=float(n_sub))
    # A zero router gives every sub-expert probability 1/n_sub; route_scale n_sub
    # makes the equal gate 1, so the routed output must be the whole expert.
    res = O.layer_forward(spec, x, np.zeros((n_sub, H)), wgu, wd, [n_sub] * T)
    ref = np.stack([neuron_sum_expert(x[t], Wg[0], Wu[0], Wd[0]) for t in range(T)])
    assert rel_err(res["out"], ref) <= 1e-12
    assert np.allclose(res["topk_w"], 1.0, rtol=0, atol=1e-15)


# ----------------------------------------------------------------------------
# P2  k = E_r with softmax, no renorm == dense gate-weighted sum
# ----------------------------------------------------------------------------

def test_p2_full_k_is_dense_softmax_mixture():
    rng = np.random.default_rng(2)
    T, H, E_r, I_sub = 4, 16, 6, 8
    x = rng.normal(size=(T, H))
    R = rng.normal(size=(E_r, H))
    wgu = rng.normal(size=(E_r, 2 * I_sub, H)) / 4
    wd = rng.normal(size=(E_r, H, I_sub)) / 3
    spec = O.LayerSpec(T=T, H=H, n_experts=E_r, n_sub=1, I_sub=I_sub, k_max=E_r)
    res = O.layer_forward(spec, x, R, wgu, wd, [E_r] * T)
    p = scipy.special.softmax(x @ R.T, axis=1)            # library softmax
    ref = np.zeros((T, H))
    for t in range(T):
        for u in range(E_r):
            ref[t] += p[t, u] * neuron_sum_expert(x[t], wgu[u, :I_sub], wgu[u, I_sub:], wd[u])
    assert rel_err(res["out"], ref) <= 1e-12


# ----------------------------------------------------------------------------
# P3  repeated-row linear gate at k = N k_orig == the unsplit layer
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("score,renorm", [("softmax", False), ("softmax", True),
                                          ("sigmoid", True), ("sigmoid", False)])
@pytest.mark.parametrize("random_partition", [False, True])
def test_p3_repeated_row_gate_reproduces_unsplit(score, renorm, random_partition):
    rng = np.random.default_rng(3)
    T, H, E, n_sub, I_sub, k_orig = 6, 16, 5, 3, 4, 2
    I = n_sub * I_sub
    x = rng.normal(size=(T, H))
    R0 = rng.normal(size=(E, H))
    Wg = rng.normal(size=(E, I, H)) / 4
    Wu = rng.normal(size=(E, I, H)) / 4
    Wd = rng.normal(size=(E, H, I)) / 3
    parts = [rng.permutation(I) for _ in range(E)] if random_partition else None
    wgu, wd = split_experts(Wg, Wu, Wd, n_sub, parts)
    R = np.repeat(R0, n_sub, axis=0)                      # MoE-Prism §III-B2 LG init
    # N-adjusted routed scaling: a gate normalised over units (softmax, or any
    # renormalisation over the selection) gives each of the n_sub copies of
    # expert e 1/n_sub of e's share, so the scale is n_sub; a raw sigmoid gives
    # every copy the full sigma(l_e), so it needs none.
    scale = 1.0 if (score == "sigmoid" and not renorm) else float(n_sub)
    spec = O.LayerSpec(T=T, H=H, n_experts=E, n_sub=n_sub, I_sub=I_sub, k_max=n_sub * k_orig,
                       score=score, renorm=renorm, route_scale=scale)
    # a per-expert logit bias is shared by the n_sub sub-experts of the expert
    bias = rng.normal(size=E)
    res = O.layer_forward(spec, x, R, wgu, wd, [n_sub * k_orig] * T, expert_bias=bias)
    ref = naive_moe(x, R0, Wg, Wu, Wd, [k_orig] * T, score=score, renorm=renorm, bias=bias)
    assert rel_err(res["out"], ref) <= 1e-12
    # the selected units are exactly the sub-experts of the top-k_orig experts
    L0 = x @ R0.T + bias[None, :]
    for t in range(T):
        top = np.argsort(-L0[t], kind="stable")[:k_orig]
        want = sorted(e * n_sub + n for e in top for n in range(n_sub))
        assert sorted(res["topk_idx"][t].tolist()) == want


# ----------------------------------------------------------------------------
# P4  routed work is linear in k
# ----------------------------------------------------------------------------

def test_p4_routed_flops_linear_in_k():
    rng = np.random.default_rng(4)
    T, H, E_r, I_sub, k_max = 9, 16, 8, 8, 5
    x = rng.normal(size=(T, H))
    R = rng.normal(size=(E_r, H))
    wgu = rng.normal(size=(E_r, 2 * I_sub, H))
    wd = rng.normal(size=(E_r, H, I_sub))
    k = rng.integers(1, k_max + 1, size=T)
    spec = O.LayerSpec(T=T, H=H, n_experts=E_r, n_sub=1, I_sub=I_sub, k_max=k_max)
    res = O.layer_forward(spec, x, R, wgu, wd, k)
    f = res["flops"]
    assert res["n_assign"] == int(k.sum())
    assert f.routed == 6 * H * I_sub * int(k.sum()) == O.routed_flops(H, I_sub, k)
    assert f.gate_up == 2 * f.down                       # expansion side is 2/3
    res2 = O.layer_forward(spec, x, R, wgu, wd, np.minimum(2 * k, k_max))
    assert res2["flops"].routed == 6 * H * I_sub * int(np.minimum(2 * k, k_max).sum())


# ----------------------------------------------------------------------------
# P5  top-k == brute force, including adversarial values
# ----------------------------------------------------------------------------

def brute_topk(row, k):
    """Selection by explicit pairwise comparisons: a beats b when a is a number
    and b is NaN, or both are numbers and a > b, or they tie (equal numbers, or
    both NaN) and a has the lower index."""
    def beats(a, b):
        la, lb = row[a], row[b]
        na, nb = math.isnan(la), math.isnan(lb)
        if na != nb:
            return nb
        if not na and la != lb:
            return la > lb
        return a < b
    left = list(range(len(row)))
    out = []
    for _ in range(k):
        best = left[0]
        for c in left[1:]:
            if beats(c, best):
                best = c
        out.append(best)
        left.remove(best)
    return out


@pytest.mark.parametrize("case", ["random", "all_equal", "signed_zero", "duplicates", "inf",
                                  "nan", "fp32_near_ties"])
def test_p5_topk_matches_brute_force(case):
    rng = np.random.default_rng(5)
    T, E_r, k_max = 12, 19, 7
    if case == "random":
        L = rng.normal(size=(T, E_r))
    elif case == "all_equal":
        L = np.full((T, E_r), 0.3)
    elif case == "signed_zero":
        L = rng.choice([-0.0, 0.0, -1.0, 1.0], size=(T, E_r))
    elif case == "duplicates":
        L = rng.choice([0.5, 0.25, -2.0], size=(T, E_r))
    elif case == "inf":
        L = rng.choice([np.inf, -np.inf, 0.0, 1.0, -0.0], size=(T, E_r))
    elif case == "nan":
        L = rng.choice([np.nan, 1.0, -1.0, 0.0, -np.inf], size=(T, E_r))
    else:
        base = np.float32(1.0)
        L = np.array([[base + np.float32(2 ** -23) * rng.integers(0, 3) for _ in range(E_r)]
                      for _ in range(T)], dtype=np.float32).astype(np.float64)
    k = rng.integers(1, k_max + 1, size=T)
    idx, flags = O.select_topk(L, k, k_max)
    for t in range(T):
        assert idx[t, :k[t]].tolist() == brute_topk(L[t].tolist(), int(k[t]))
        assert (idx[t, k[t]:] == -1).all()
    assert bool(flags & O.FLAG_NONFINITE) == bool((~np.isfinite(L)).any())


def test_p5_k_range_flag():
    L = np.zeros((3, 4))
    _, flags = O.select_topk(L, [1, 0, 2], 2)
    assert flags & O.FLAG_K_RANGE
    _, flags = O.select_topk(L, [1, 3, 2], 2)
    assert flags & O.FLAG_K_RANGE
    _, flags = O.select_topk(L, [1, 2, 2], 2)
    assert flags == 0


# ----------------------------------------------------------------------------
# P6  permutation: bijection, ordering, brute force enumeration
# ----------------------------------------------------------------------------

def test_p6_permutation_properties_and_brute_force():
    rng = np.random.default_rng(6)
    for trial in range(50):
        T = int(rng.integers(1, 5))
        E_r = int(rng.integers(1, 9))
        k_max = int(rng.integers(1, E_r + 1))
        k = rng.integers(1, k_max + 1, size=T)
        idx = np.full((T, k_max), -1, dtype=np.int32)
        for t in range(T):
            idx[t, :k[t]] = rng.permutation(E_r)[:k[t]]
        counts, offsets, st, inv = O.permute(idx, k, E_r)
        n = int(k.sum())
        assert counts.sum() == n and offsets[-1] == n and (np.diff(offsets) == counts).all()
        pos = sorted(int(inv[t, j]) for t in range(T) for j in range(k[t]))
        assert pos == list(range(n))                       # bijection onto [0, n)
        # brute force: walk units in order, tokens in order
        want = [t for u in range(E_r) for t in range(T) if u in idx[t, :k[t]].tolist()]
        assert st.tolist() == want
        for t in range(T):
            for j in range(k[t]):
                r = inv[t, j]
                assert st[r] == t and offsets[idx[t, j]] <= r < offsets[idx[t, j] + 1]
            assert (inv[t, k[t]:] == -1).all()


# ----------------------------------------------------------------------------
# P7  gate weights: probabilities sum to 1, renormalised weights to route_scale
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("score", ["softmax", "sigmoid"])
def test_p7_gate_sums(score):
    rng = np.random.default_rng(7)
    T, E_r = 10, 13
    L = rng.normal(size=(T, E_r)) * 3
    full = np.tile(np.arange(E_r), (T, 1)).astype(np.int32)
    if score == "softmax":
        w = O.gate_weights(L, full, [E_r] * T, score, False, 1.0)
        assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        # each entry equals the library softmax
        assert np.allclose(w, scipy.special.softmax(L, axis=1), rtol=1e-14, atol=0)
    else:
        w = O.gate_weights(L, full, [E_r] * T, score, False, 1.0)
        assert np.allclose(w, scipy.special.expit(L), rtol=1e-14, atol=0)
    k = rng.integers(1, 6, size=T)
    idx, _ = O.select_topk(L, k, 5)
    w = O.gate_weights(L, idx, k, score, True, 2.5)
    assert np.allclose(w.sum(axis=1), 2.5, rtol=1e-14)
    for t in range(T):
        assert (w[t, k[t]:] == 0).all()


# ----------------------------------------------------------------------------
# P8  closed-form one-hot layer (golden fixture)
# ----------------------------------------------------------------------------

def _load_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_p8_onehot_layer_matches_golden():
    H = 4
    e = np.eye(H)
    wgu = np.zeros((2, 2, H))
    wd = np.zeros((2, H, 1))
    wgu[0, 0], wgu[0, 1], wd[0][:, 0] = e[0], e[1], e[2]
    wgu[1, 0], wgu[1, 1], wd[1][:, 0] = e[1], e[3], 2 * e[0]
    x = np.array([[1.0, 2.0, -1.0, 0.5]])
    logits = np.array([[0.0, math.log(3.0)]])
    f0 = 1.0 * _sig(1.0) * 2.0
    f1 = 2.0 * _sig(2.0) * 0.5 * 2.0
    rows = _load_rows("onehot_swiglu.txt")
    assert len(rows) == 5
    for score, renorm, k, *vals in rows:
        renorm, k = bool(int(renorm)), int(k)
        spec = O.LayerSpec(T=1, H=H, n_experts=1, n_sub=2, I_sub=1, k_max=2, score=score,
                           renorm=renorm)
        res = O.layer_forward(spec, x, np.zeros((2, H)), wgu, wd, [k], logits=logits)
        want = np.array([float(v) for v in vals])
        # the fixture itself agrees with the closed form
        if score == "softmax":
            s = [0.25, 0.75]
        else:
            s = [0.5, 0.75]
        sel = [1] if k == 1 else [1, 0]
        tot = sum(s[u] for u in sel)
        cf = np.zeros(H)
        for u in sel:
            w = s[u] / tot if renorm else s[u]
            if u == 0:
                cf[2] += w * f0
            else:
                cf[0] += w * f1
        assert np.allclose(cf, want, rtol=1e-15, atol=0)
        assert np.allclose(res["out"][0], want, rtol=1e-15, atol=0)


# ----------------------------------------------------------------------------
# P9  coarse execution budget k_exec = N ceil(k / N)
# ----------------------------------------------------------------------------

def test_p9_coarse_k_golden():
    for N, kq, ke in _load_rows("k_exec_rounding.txt"):
        assert O.coarse_k(int(kq), int(N)) == int(ke)


def test_p9_coarse_split_equals_unsplit_rounded_up():
    rng = np.random.default_rng(9)
    T, H, E, n_sub, I_sub = 5, 12, 4, 4, 3
    I = n_sub * I_sub
    x = rng.normal(size=(T, H))
    R0 = rng.normal(size=(E, H))
    Wg = rng.normal(size=(E, I, H)) / 3
    Wu = rng.normal(size=(E, I, H)) / 3
    Wd = rng.normal(size=(E, H, I)) / 3
    wgu, wd = split_experts(Wg, Wu, Wd, n_sub)
    R = np.repeat(R0, n_sub, axis=0)
    k_qos = np.array([1, 3, 4, 6, 7])
    k_exec = np.array([O.coarse_k(int(k), n_sub) for k in k_qos])
    spec = O.LayerSpec(T=T, H=H, n_experts=E, n_sub=n_sub, I_sub=I_sub, k_max=int(k_exec.max()),
                       route_scale=float(n_sub))
    res = O.layer_forward(spec, x, R, wgu, wd, k_exec)
    ref = naive_moe(x, R0, Wg, Wu, Wd, [int(math.ceil(k / n_sub)) for k in k_qos])
    assert rel_err(res["out"], ref) <= 1e-12


# ----------------------------------------------------------------------------
# P10  tiny end-to-end layer vs the naive formulation (bias included)
# ----------------------------------------------------------------------------

def test_p10_tiny_layer_vs_naive():
    rng = np.random.default_rng(10)
    T, H, E, I_sub, k_max = 6, 32, 8, 16, 4
    x = rng.normal(size=(T, H))
    R = rng.normal(size=(E, H)) / math.sqrt(H)
    bias = rng.normal(size=E)
    Wg = rng.normal(size=(E, I_sub, H)) / math.sqrt(H)
    Wu = rng.normal(size=(E, I_sub, H)) / math.sqrt(H)
    Wd = rng.normal(size=(E, H, I_sub)) / math.sqrt(I_sub)
    wgu, wd = split_experts(Wg, Wu, Wd, 1)
    k = rng.integers(1, k_max + 1, size=T)
    for score, renorm in [("softmax", False), ("softmax", True), ("sigmoid", True)]:
        spec = O.LayerSpec(T=T, H=H, n_experts=E, n_sub=1, I_sub=I_sub, k_max=k_max,
                           score=score, renorm=renorm, route_scale=1.5)
        res = O.layer_forward(spec, x, R, wgu, wd, k, expert_bias=bias)
        ref = naive_moe(x, R, Wg, Wu, Wd, k, score=score, renorm=renorm, scale=1.5, bias=bias)
        assert rel_err(res["out"], ref) <= 1e-12


def test_shared_expert_adds_with_weight_one():
    rng = np.random.default_rng(11)
    T, H, E, I_sub, I_sh = 3, 8, 4, 4, 6
    x = rng.normal(size=(T, H))
    R = rng.normal(size=(E, H))
    wgu = rng.normal(size=(E, 2 * I_sub, H))
    wd = rng.normal(size=(E, H, I_sub))
    sgu = rng.normal(size=(2 * I_sh, H))
    sd = rng.normal(size=(H, I_sh))
    spec = O.LayerSpec(T=T, H=H, n_experts=E, n_sub=1, I_sub=I_sub, k_max=2, score="sigmoid",
                       renorm=True, I_shared=I_sh)
    res = O.layer_forward(spec, x, R, wgu, wd, [2] * T, w_shared_gate_up=sgu, w_shared_down=sd)
    base = O.layer_forward(O.LayerSpec(T=T, H=H, n_experts=E, n_sub=1, I_sub=I_sub, k_max=2,
                                       score="sigmoid", renorm=True), x, R, wgu, wd, [2] * T)
    sh = np.stack([neuron_sum_expert(x[t], sgu[:I_sh], sgu[I_sh:], sd) for t in range(T)])
    assert rel_err(res["out"] - base["out"], sh) <= 1e-12


def test_bf16_bit_conversion_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x8000, 0x7F80, 0x4049, 0x0001], dtype=np.uint16)
    v = O.bf16_to_f64(bits)
    assert v[0] == 1.0 and v[1] == -1.0 and v[2] == 0.0 and math.copysign(1, v[3]) < 0
    assert math.isinf(v[4]) and v[5] == 3.140625 and v[6] == 2.0 ** -133


def test_distinct_units_counts_nonzero_units():
    assert O.distinct_units(np.array([0, 3, 0, 1, 7])) == 3
    assert O.distinct_units(np.zeros(5, dtype=np.int32)) == 0
    # from a permutation: every selected unit is counted once
    idx = np.array([[2, 0, -1], [2, 5, 1]], dtype=np.int32)
    counts, *_ = O.permute(idx, [2, 3], 6)
    assert O.distinct_units(counts) == 4


def test_budget_generators_and_modes():
    """Eq. (7) draws stay in [1, k_max] and follow the mean; the comparison
    modes give the batch maximum everywhere, or n_sub * ceil(k / n_sub)."""
    import torch
    from aware_moe_expert_gb300.inputs import apply_k_mode, draw_k_normal
    k = draw_k_normal(20000, 6.0, 2.0, 8, seed=3)
    assert int(k.min()) >= 1 and int(k.max()) <= 8
    assert abs(float(k.double().mean()) - 5.85) < 0.1   # E[clip(round(N(6,4)),1,8)] ~ 5.85
    base = torch.tensor([1, 2, 3, 4, 5, 7, 8], dtype=torch.int32)
    assert apply_k_mode(base, "batch_max", 4, 8).tolist() == [8] * 7
    assert apply_k_mode(base, "coarse", 4, 8).tolist() == [4, 4, 4, 4, 8, 8, 8]
    assert apply_k_mode(base, "coarse", 2, 7).tolist() == [2, 2, 4, 4, 6, 7, 7]
    assert [O.coarse_k(int(v), 4) for v in base] == [4, 4, 4, 4, 8, 8, 8]


def test_several_routings_at_once_match_the_naive_layer():
    """layer_forward_routings: every routing it returns equals the naive
    formulation run on that routing's own logits (the float64 logits of the
    router, or perturbed fp32 logits that select differently for some
    tokens), shared expert included."""
    rng = np.random.default_rng(14)
    T, H, E, I_sub, k_max, I_sh = 7, 16, 6, 8, 3, 4
    x = rng.normal(size=(T, H))
    R = rng.normal(size=(E, H)) / math.sqrt(H)
    Wg = rng.normal(size=(E, I_sub, H)) / math.sqrt(H)
    Wu = rng.normal(size=(E, I_sub, H)) / math.sqrt(H)
    Wd = rng.normal(size=(E, H, I_sub)) / math.sqrt(I_sub)
    sgu = rng.normal(size=(2 * I_sh, H))
    sd = rng.normal(size=(H, I_sh))
    wgu, wd = split_experts(Wg, Wu, Wd, 1)
    k = rng.integers(1, k_max + 1, size=T)
    L64 = x @ R.T
    L32 = (L64 + rng.normal(size=L64.shape) * 0.3).astype(np.float32)
    spec = O.LayerSpec(T=T, H=H, n_experts=E, n_sub=1, I_sub=I_sub, k_max=k_max,
                       I_shared=I_sh)
    r64, r32 = O.layer_forward_routings(spec, x, R, wgu, wd, k, logits_list=(None, L32),
                                        w_shared_gate_up=sgu, w_shared_down=sd)
    sh = np.stack([neuron_sum_expert(x[t], sgu[:I_sh], sgu[I_sh:], sd) for t in range(T)])
    for res, L in ((r64, L64), (r32, L32.astype(np.float64))):
        ref = naive_moe_from_logits(x, L, Wg, Wu, Wd, k)
        assert rel_err(res["out"], ref + sh) <= 1e-12
    assert not np.array_equal(r64["topk_idx"], r32["topk_idx"])   # the routings differ
