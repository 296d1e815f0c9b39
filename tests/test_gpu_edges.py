"""Edge cases of the whole layer against the oracle.

The largest routing budget the ABI accepts: k_max = 32 over E_r = 256 units,
every token at k_t = 32 (MoE-Prism §III-C1: a request's budget can be any
number of sub-experts up to the layer's maximum).

The Qwen3-30B-A3B-shaped decode layer (H 2048, 128 experts x 2 sub-experts of
384) at four token counts exercises every kernel family at that budget: the
cluster router with the permutation in the same launch and the fused decode
FFN (T = 8), the decode FFN with the one-CTA permutation (T = 64) and with
the bitmap permutation (T = 300), and the tensor-core router, the top-k
kernel writing the bitmap and the prefill grouped GEMMs (T = 1024, where
T * k_max exceeds 64 * E_r).  Every token is compared with the oracle up to
T = 64; above, a seeded sample with the first and last token.

The degenerate layers with a single expert (one unit at k = 1; one expert
split four ways, all selected), every unit selected by every token (k =
E_r), a shared expert at decode token counts, and 9 to 16 tokens (the fused
decode FFN's 16-token chunks gathering their own rows).
"""
from dataclasses import replace

import numpy as np
import pytest

from aware_moe_expert_gb300 import binding as B
from aware_moe_expert_gb300 import workloads as WL
from test_gpu_layer import _compare, _run_layer

pytestmark = pytest.mark.gpu

K32 = replace(WL.QWEN_DECODE, name="qwen3-30b-a3b-decode-k32", k_max=32, k_choices=(32,))


@pytest.mark.parametrize("T", [8, 64, 300, 1024])
def test_layer_at_k_max_32(T):
    wl, d, desc, out, Lg, idx = _run_layer(K32, T=T)
    k = d["k_per_token"].cpu().numpy()
    assert int(k.min()) == 32 and int(k.max()) == 32
    # every token selected 32 distinct units
    sel = idx.cpu().numpy()
    assert all(len(set(row.tolist())) == 32 for row in sel)
    if T <= 64:
        tokens = np.arange(T)
    else:
        rng = np.random.default_rng(T)
        tokens = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 48, replace=False)]))
    fro, n_tied = _compare(wl, d, desc, out, Lg, idx, tokens)
    assert fro <= 5e-3


@pytest.mark.parametrize("path", [B.PATH_DECODE, B.PATH_PREFILL])
def test_layer_at_k_max_32_both_families(path):
    """The same budget forced onto each grouped-GEMM family (T = 64)."""
    wl, d, desc, out, Lg, idx = _run_layer(K32, T=64, path=path)
    _compare(wl, d, desc, out, Lg, idx, np.arange(64))


# The degenerate layer: one routing unit, k = 1, so every token's gate is 1
# (softmax over a single logit) and the layer is one dense SwiGLU FFN.
ONE_UNIT = replace(WL.TINY, name="one-unit-h256-i128", n_experts=1, n_sub=1, k_max=1,
                   k_choices=(1,))
# One expert split into four sub-experts, all four selected by every token:
# the gate-weighted sum of the slices (MoE-Prism §III-B1 Eq. (3) with
# softmax gates).
ONE_EXPERT_SPLIT = replace(WL.TINY, name="one-expert-x4-h256-i128", n_experts=1, n_sub=4,
                           k_max=4, k_choices=(4,))


@pytest.mark.parametrize("wl", [ONE_UNIT, ONE_EXPERT_SPLIT], ids=lambda w: w.name)
@pytest.mark.parametrize("T", [1, 8, 200])
def test_layer_with_a_single_expert(wl, T):
    wl, d, desc, out, Lg, idx = _run_layer(wl, T=T)
    _compare(wl, d, desc, out, Lg, idx, np.arange(T))


# DeepSeek-V3-shaped layer (H 7168, I_sub 2048, a shared expert, sigmoid
# scores renormalised over the selection) with 16 routed experts, at decode
# token counts: the shared expert's dense GEMMs on a handful of rows and the
# fused decode FFN at H = 7168.
DEEPSEEK_SMALL = replace(WL.DEEPSEEK_PREFILL, name="deepseek-v3-shape-e16-decode", n_experts=16,
                         tokens_per_request=1, phase="decode")


@pytest.mark.parametrize("T", [1, 5, 64])
def test_layer_shared_expert_at_decode_sizes(T):
    wl, d, desc, out, Lg, idx = _run_layer(DEEPSEEK_SMALL, T=T)
    _compare(wl, d, desc, out, Lg, idx, np.arange(T))


@pytest.mark.parametrize("T,path", [(128, B.PATH_AUTO), (300, B.PATH_AUTO), (257, B.PATH_PREFILL),
                                    (700, B.PATH_AUTO)])
def test_layer_shared_expert_at_prefill_sizes(T, path):
    """The shared expert's dense GEMMs on single-CTA tiles (up to 600 rows)
    and on CTA pairs (700 rows), with ragged last tiles, next to the routed
    GEMMs at H = 7168 (routed down on CTA pairs: I_sub = 2048): every token
    against the oracle."""
    wl, d, desc, out, Lg, idx = _run_layer(DEEPSEEK_SMALL, T=T, path=path)
    _compare(wl, d, desc, out, Lg, idx, np.arange(T))


# Every token selects every unit (k = E_r = 32): the dense gate-weighted
# mixture of all sub-experts (MoE-Prism §II, Eq. (2) with k = all), every
# unit serving all T tokens.
ALL_UNITS = replace(WL.TINY, name="all-units-e8x4-h256", n_experts=8, n_sub=4, k_max=32,
                    k_choices=(32,))


@pytest.mark.parametrize("T", [1, 64, 200])
def test_layer_with_every_unit_selected(T):
    wl, d, desc, out, Lg, idx = _run_layer(ALL_UNITS, T=T)
    sel = np.sort(idx.cpu().numpy(), axis=1)
    assert (sel == np.arange(32)[None, :]).all()
    _compare(wl, d, desc, out, Lg, idx, np.arange(T))


@pytest.mark.parametrize("name,T", [("qwen_decode", 9), ("qwen_decode", 12), ("qwen_decode", 16),
                                    ("mixtral_decode", 16), ("tiny", 9)])
def test_layer_between_the_cluster_router_and_64_token_chunks(name, T):
    """9 to 16 tokens: routed and permuted by the general kernels (more than
    one cluster's eight tokens), then the fused decode FFN with 16-token
    chunks that gathers its token rows from x itself."""
    wl, d, desc, out, Lg, idx = _run_layer(WL.ALL[name], T=T)
    _compare(wl, d, desc, out, Lg, idx, np.arange(T))
