"""The layer at the largest routing budget the ABI accepts: k_max = 32 over
E_r = 256 units, every token at k_t = 32 (MoE-Prism §III-C1: a request's
budget can be any number of sub-experts up to the layer's maximum).

The Qwen3-30B-A3B-shaped decode layer (H 2048, 128 experts x 2 sub-experts of
384) at four token counts exercises every kernel family at that budget: the
cluster router with the permutation in the same launch and the fused decode
FFN (T = 8), the decode FFN with the one-CTA permutation (T = 64) and with
the bitmap permutation (T = 300), and the tensor-core router, the top-k
kernel writing the bitmap and the prefill grouped GEMMs (T = 1024, where
T * k_max exceeds 64 * E_r).  Every token is compared with the oracle up to
T = 64; above, a seeded sample with the first and last token.
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
