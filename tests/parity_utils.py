"""Shared helpers of the parity tests: the stated tolerance, oracle adapters
and the near-tie rule for routing from independently computed logits."""
from __future__ import annotations

import numpy as np
import torch

from aware_moe_expert_gb300 import binding as B
from aware_moe_expert_gb300.inputs import bf16_bits
from oracle import moe_oracle as O

# Layer output tolerance: per element |d| <= ATOL + RTOL*|ref|, and relative
# Frobenius error <= FRO over the compared tokens.
ATOL, RTOL, FRO = 1e-2, 1e-2, 5e-3
# Gate weights of the same fp32 logits: fp32 softmax/sigmoid with expf
# (<= 2 ulp), a sum of <= 256 positive terms in fp32 and one division; the
# relative error is bounded by about (E_r + 16) * 2^-24 <= 1.7e-5.
W_RTOL = 2e-5


def spec_of(desc: B.LayerDesc, T=None) -> O.LayerSpec:
    return O.LayerSpec(T=desc.T if T is None else T, H=desc.H, n_experts=desc.n_experts,
                       n_sub=desc.n_sub, I_sub=desc.I_sub, k_max=desc.k_max, score=desc.score,
                       renorm=bool(desc.renorm), route_scale=desc.route_scale,
                       I_shared=desc.I_shared)


def assert_close_layer(got: np.ndarray, ref: np.ndarray, what: str = "out"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(got - ref)
    lim = ATOL + RTOL * np.abs(ref)
    bad = d > lim
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements outside |d| <= {ATOL} + {RTOL}|ref|"
                           f"; worst d={d.max():.3e}; fro={fro:.3e}")
    assert fro <= FRO, f"{what}: relative Frobenius error {fro:.3e} > {FRO}"
    return fro


def to_np_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def unit_fetch(w: torch.Tensor):
    """Oracle weight accessor: one unit's bf16 bit patterns copied to host."""
    return lambda u: bf16_bits(w[u])


def tie_safe_tokens(L64: np.ndarray, gpu_idx: np.ndarray, k: np.ndarray, delta: np.ndarray):
    """Tokens whose selection is decided with margin.

    The GPU selects on fp32 logits accumulated in its own order; the oracle on
    float64 logits.  Where the oracle's k-th and (k+1)-th logits are closer
    than ``delta`` (twice the measured logit error of that token), either
    selection is a correct result.  Returns (ok_mask, n_tied): ok_mask marks
    tokens whose GPU selection equals the oracle's; a token may differ only if
    it is a near tie, and then every unit where the two selections differ must
    lie within delta of the oracle's selection boundary.
    """
    T = L64.shape[0]
    ok = np.ones(T, dtype=bool)
    n_tied = 0
    for t in range(T):
        kt = int(k[t])
        order = O.selection_order(L64[t])
        want = set(order[:kt].tolist())
        got = set(int(u) for u in gpu_idx[t, :kt])
        if want == got:
            continue
        ok[t] = False
        n_tied += 1
        boundary = 0.5 * (L64[t, order[kt - 1]] + (L64[t, order[kt]] if kt < len(order)
                                                   else L64[t, order[kt - 1]]))
        for u in want.symmetric_difference(got):
            assert abs(L64[t, u] - boundary) <= delta[t], (
                f"token {t}: selections differ at unit {u} by more than a near tie "
                f"(|L-boundary|={abs(L64[t, u] - boundary):.3e} > {delta[t]:.3e})")
    return ok, n_tied
