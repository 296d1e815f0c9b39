"""GPU parity of path-composed execution with source-grouped reuse
(moe_layer_forward_paths) against the fp64 oracle (oracle/pcomoe.py).

Paths come from the GPU's own routing through the seeded recipes of the
input generator (consecutive slots share a source; or share a target; or a
path repeats); both sides run the same paths.  Outputs are compared in the
stated layer tolerance, on the decode kernels and on the prefill kernels
(forced by desc.path), with diagonal paths (the plain layer) as a special
case.
"""
import numpy as np
import pytest
import torch

from aware_moe_expert_gb300 import binding as B
from aware_moe_expert_gb300 import workloads as WL
from aware_moe_expert_gb300.inputs import make_layer_inputs, make_paths, bf16_bits
from oracle import moe_oracle as O
from oracle import pcomoe as P
from parity_utils import assert_close_layer, unit_fetch

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(wl, path, diagonal=False, n_check=None, mode="share_source"):
    d = make_layer_inputs(wl, DEV)
    desc = B.desc_for(wl, expert_bias=d["expert_bias"], w_shared_gate_up=d.get("w_shared_gate_up"),
                      w_shared_down=d.get("w_shared_down"))
    desc.path = path
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx = torch.empty(wl.T, wl.k_max, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.k_max, dtype=torch.float32, device=DEV)
    B.check(B.moe_route(desc, d["x"], d["router_w"], None, d["k_per_token"], None, idx, w, st, ws))
    src, tgt, beta = make_paths(idx, w, mode)
    if diagonal:
        src = tgt.clone()
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)
    B.check(B.moe_layer_forward_paths(desc, d["x"], d["w_gate_up"], d["w_down"], src, tgt, beta,
                                      d["k_per_token"], out, st, ws), "moe_layer_forward_paths")
    code = B.moe_get_device_status(st)
    assert code == 0, B.STATUS_NAMES[code]
    tokens = np.arange(wl.T) if n_check is None else np.unique(
        np.r_[0, wl.T - 1, np.random.default_rng(1).choice(wl.T, n_check, replace=False)])
    x = O.bf16_to_f64(bf16_bits(d["x"]))[tokens]
    wgu, wd = unit_fetch(d["w_gate_up"]), unit_fetch(d["w_down"])
    cache_g, cache_d = {}, {}

    def g(u):
        if u not in cache_g:
            cache_g[u] = O.bf16_to_f64(wgu(u))
        return cache_g[u]

    def dn(u):
        if u not in cache_d:
            cache_d[u] = O.bf16_to_f64(wd(u))
        return cache_d[u]
    k = d["k_per_token"].cpu().numpy()[tokens]
    sh = {}
    if wl.I_shared:
        sh = dict(w_shared_gate_up=O.bf16_to_f64(bf16_bits(d["w_shared_gate_up"])),
                  w_shared_down=O.bf16_to_f64(bf16_bits(d["w_shared_down"])))
    ref, n_exp = P.paths_forward(x, g, dn, src.cpu().numpy()[tokens], tgt.cpu().numpy()[tokens],
                                 beta.cpu().numpy()[tokens], k, **sh)
    assert_close_layer(out.to(torch.float64).cpu().numpy()[tokens], ref, f"{wl.name} paths")
    t_np = tgt.cpu().numpy()[tokens]
    n_proj = sum(len(set(t_np[i, :k[i]].tolist())) for i in range(len(tokens)))
    return n_exp, int(k.sum()), n_proj


@pytest.mark.parametrize("name,T", [("tiny", None), ("qwen_decode", 8), ("qwen_decode", 64),
                                    ("mixtral_decode", None)])
@pytest.mark.parametrize("path", [B.PATH_DECODE, B.PATH_PREFILL])
def test_paths_match_oracle(name, T, path):
    wl = WL.ALL[name] if T is None else WL.ALL[name].with_T(T)
    n_exp, n_paths, _ = _run(wl, path)
    assert n_exp < n_paths          # the recipe shares sources, so fewer expansions


@pytest.mark.parametrize("mode", ["share_target", "duplicate"])
@pytest.mark.parametrize("name,T", [("tiny", None), ("qwen_decode", 8), ("qwen_decode", 64),
                                    ("mixtral_decode", None), ("qwen_decode", 300)])
@pytest.mark.parametrize("path", [B.PATH_DECODE, B.PATH_PREFILL])
def test_paths_sharing_a_target_match_oracle(name, T, path, mode):
    """Several paths of a token into one target (and, with 'duplicate', the
    same path twice): one projection per distinct target, fed the weighted
    sum of the paths' expansions."""
    wl = WL.ALL[name] if T is None else WL.ALL[name].with_T(T)
    n_exp, n_paths, n_proj = _run(wl, path, mode=mode)
    assert n_proj < n_paths         # the recipe shares targets, so fewer projections


def test_diagonal_paths_are_the_plain_layer():
    n_exp, n_paths, n_proj = _run(WL.TINY, B.PATH_AUTO, diagonal=True)
    assert n_exp == n_paths == n_proj


@pytest.mark.parametrize("mode", ["share_source", "share_target"])
@pytest.mark.parametrize("name,T", [("qwen_prefill", 2048), ("deepseek_prefill", 1024)])
def test_prefill_sized_paths_sampled(name, T, mode):
    """Prefill kernels at model sizes (the DeepSeek-V3 shape adds its shared
    expert), a seeded sample of tokens against the oracle."""
    n_exp, n_paths, n_proj = _run(WL.ALL[name].with_T(T), B.PATH_AUTO, n_check=32, mode=mode)
    assert min(n_exp, n_proj) < n_paths


def test_out_of_range_target_is_reported():
    """A unit index outside [0, E_r) is reported (MOE_ERR_BAD_INDEX), not read."""
    wl = WL.TINY.with_T(4)
    d = make_layer_inputs(wl, DEV)
    desc = B.desc_for(wl, expert_bias=d["expert_bias"])
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    k = torch.full((4,), 2, dtype=torch.int32, device=DEV)
    src = torch.tensor([[0, 1]] * 4, dtype=torch.int32, device=DEV)
    tgt = torch.tensor([[5, wl.E_r]] * 4, dtype=torch.int32, device=DEV)
    beta = torch.ones(4, 2, device=DEV)
    src = torch.nn.functional.pad(src, (0, wl.k_max - 2), value=-1)
    tgt = torch.nn.functional.pad(tgt, (0, wl.k_max - 2), value=-1)
    beta = torch.nn.functional.pad(beta, (0, wl.k_max - 2))
    out = torch.empty(4, wl.H, dtype=torch.bfloat16, device=DEV)
    B.check(B.moe_layer_forward_paths(desc, d["x"], d["w_gate_up"], d["w_down"], src, tgt, beta,
                                      k, out, st, ws))
    assert B.moe_get_device_status(st) == 8   # MOE_ERR_BAD_INDEX
