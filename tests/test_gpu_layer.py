"""End-to-end parity of moe_layer_forward on the five synthetic workloads.

Two comparisons per case, both against the fp64 oracle:
  1. on the GPU's own fp32 logits (moe_route's logits_out, the same kernels
     as inside the layer): the oracle's selection must equal the GPU's bit
     for bit and EVERY compared token's output must be within the layer
     tolerance, no token left out;
  2. on the oracle's own float64 logits: a token whose k-th and (k+1)-th
     logits nearly tie may legitimately select a different unit; such tokens
     must be genuine near ties (checked), are counted, and are left out of
     this mode's element comparison only.
Small workloads compare every token; the two large prefill workloads compare
whole 512-token requests plus a seeded sample and the first and last token
(the oracle runs on those tokens: tokens are independent), plus properties
that hold at any size (routing and permutation bit-exact from
generator-given logits).
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from aware_moe_expert_gb300 import binding as B
from aware_moe_expert_gb300 import workloads as WL
from aware_moe_expert_gb300.inputs import make_layer_inputs, make_logits, bf16_bits
from oracle import moe_oracle as O
from parity_utils import assert_close_layer, spec_of, unit_fetch, tie_safe_tokens

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run_layer(wl, T=None, path=B.PATH_AUTO):
    wl = wl if T is None else wl.with_T(T)
    d = make_layer_inputs(wl, DEV)
    desc = B.desc_for(wl, expert_bias=d["expert_bias"], w_shared_gate_up=d.get("w_shared_gate_up"),
                      w_shared_down=d.get("w_shared_down"))
    desc.path = path
    layer = B.MoeLayer(desc, DEV)
    out = layer.forward(d["x"], d["router_w"], d["w_gate_up"], d["w_down"], d["k_per_token"])
    code = layer.device_status()
    assert code == 0, B.STATUS_NAMES[code]
    # the GPU's own logits and selection (same kernels as inside the layer)
    Lg = torch.empty(wl.T, wl.E_r, dtype=torch.float32, device=DEV)
    idx = torch.empty(wl.T, wl.k_max, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.k_max, dtype=torch.float32, device=DEV)
    B.check(B.moe_route(desc, d["x"], d["router_w"], None, d["k_per_token"], Lg, idx, w,
                        layer.status, layer.workspace))
    assert layer.device_status() == 0
    return wl, d, desc, out, Lg, idx


def _compare(wl, d, desc, out, Lg, idx, tokens):
    tokens = np.asarray(tokens)
    x_s = bf16_bits(d["x"][torch.as_tensor(tokens, device=DEV)])
    k_s = d["k_per_token"].cpu().numpy()[tokens]
    bias = None if d["expert_bias"] is None else d["expert_bias"].cpu().numpy()
    spec = spec_of(desc, T=len(tokens))
    Lg_s = Lg.cpu().numpy()[tokens]
    idx_s = idx.cpu().numpy()[tokens]
    ref64, ref32 = O.layer_forward_routings(
        spec, x_s, bf16_bits(d["router_w"]), unit_fetch(d["w_gate_up"]), unit_fetch(d["w_down"]),
        k_s, expert_bias=bias, logits_list=(None, Lg_s),
        w_shared_gate_up=(bf16_bits(d["w_shared_gate_up"]) if wl.I_shared else None),
        w_shared_down=(bf16_bits(d["w_shared_down"]) if wl.I_shared else None))
    got = out.to(torch.float64).cpu().numpy()[tokens]
    # 1. the GPU's fp32 logits: same selection, every token within tolerance
    np.testing.assert_array_equal(ref32["topk_idx"], idx_s)
    fro = assert_close_layer(got, ref32["out"], f"{wl.name} (GPU logits)")
    # 2. float64 logits: near ties counted and left out of this mode only
    L64 = ref64["logits"]
    delta = 2.0 * np.abs(Lg_s.astype(np.float64) - L64).max(axis=1) + 1e-7
    ok, n_tied = tie_safe_tokens(L64, idx_s, k_s, delta)
    assert n_tied <= max(2, len(tokens) // 100), f"{n_tied} near-tie tokens"
    assert_close_layer(got[ok], ref64["out"][ok], f"{wl.name} (fp64 logits)")
    return fro, n_tied


@pytest.mark.parametrize("name", ["tiny", "mixtral_decode"])
def test_layer_all_tokens(name):
    wl, d, desc, out, Lg, idx = _run_layer(WL.ALL[name])
    _compare(wl, d, desc, out, Lg, idx, np.arange(wl.T))


@pytest.mark.parametrize("path", [B.PATH_PREFILL, B.PATH_DECODE])
@pytest.mark.parametrize("name,T", [("tiny", None), ("qwen_decode", 64), ("mixtral_decode", None)])
def test_layer_both_gemm_paths(name, T, path):
    """The prefill-tile and decode swap-AB kernels both match the oracle."""
    wl, d, desc, out, Lg, idx = _run_layer(WL.ALL[name], T=T, path=path)
    _compare(wl, d, desc, out, Lg, idx, np.arange(wl.T))


@pytest.mark.parametrize("T", WL.QWEN_DECODE_T)
def test_layer_qwen_decode_sweep(T):
    wl, d, desc, out, Lg, idx = _run_layer(WL.QWEN_DECODE, T=T)
    tokens = np.arange(T) if T <= 256 else np.random.default_rng(T).choice(T, 256, replace=False)
    _compare(wl, d, desc, out, Lg, idx, np.sort(tokens))


@pytest.mark.parametrize("name,request_idx,n_sample", [("qwen_prefill", 5, 64),
                                                      ("deepseek_prefill", 0, 32)])
def test_layer_prefill_sampled(name, request_idx, n_sample):
    """One whole 512-token request, a seeded sample of the other tokens, and
    the first and last token of the batch (the ragged tail)."""
    wl, d, desc, out, Lg, idx = _run_layer(WL.ALL[name])
    rng = np.random.default_rng(12345)
    req = np.arange(request_idx * wl.tokens_per_request, (request_idx + 1) * wl.tokens_per_request)
    tokens = np.unique(np.concatenate([[0, wl.T - 1], req,
                                       rng.choice(wl.T, n_sample, replace=False)]))
    assert len(tokens) >= wl.tokens_per_request + 1
    _compare(wl, d, desc, out, Lg, idx, tokens)


@pytest.mark.parametrize("name", ["qwen_prefill", "deepseek_prefill"])
def test_full_size_routing_and_permutation_bit_exact(name):
    """At full size: top-k, gates and the permutation from generator-given
    logits (the layer's own launch shapes for these steps)."""
    wl = WL.ALL[name]
    desc = B.desc_for(wl)
    desc.I_shared = 0          # routing and permutation do not involve the shared expert
    L = make_logits(wl.T, wl.E_r, DEV, seed=wl.seed)
    from aware_moe_expert_gb300.inputs import draw_k
    k = draw_k(wl, DEV)
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx = torch.empty(wl.T, wl.k_max, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.k_max, dtype=torch.float32, device=DEV)
    counts = torch.empty(wl.E_r, dtype=torch.int32, device=DEV)
    offsets = torch.empty(wl.E_r + 1, dtype=torch.int32, device=DEV)
    st_tok = torch.empty(wl.T * wl.k_max, dtype=torch.int32, device=DEV)
    inv = torch.empty(wl.T * wl.k_max, dtype=torch.int32, device=DEV)
    B.check(B.moe_route(desc, None, None, L, k, None, idx, w, st, ws))
    B.check(B.moe_permute(desc, idx, k, counts, offsets, st_tok, inv, st, ws))
    assert B.moe_get_device_status(st) == 0
    Ln, kn = L.cpu().numpy(), k.cpu().numpy()
    want_idx, _ = O.select_topk(Ln, kn, wl.k_max)
    np.testing.assert_array_equal(idx.cpu().numpy(), want_idx)
    wc, wo, wst, winv = O.permute(want_idx, kn, wl.E_r)
    np.testing.assert_array_equal(offsets.cpu().numpy(), wo)
    np.testing.assert_array_equal(st_tok.cpu().numpy()[: int(wo[-1])], wst)
    np.testing.assert_array_equal(inv.cpu().numpy().reshape(wl.T, wl.k_max), winv)
    assert int(wo[-1]) == int(kn.sum())


@pytest.mark.parametrize("name,T", [("tiny", None), ("qwen_decode", 64), ("qwen_decode", 256),
                                    ("qwen_decode", 300), ("mixtral_decode", None),
                                    ("qwen_decode", 128), ("qwen_decode", 129),
                                    ("qwen_decode", 1), ("qwen_decode", 8), ("mixtral_decode", 5),
                                    ("tiny", 7), ("tiny_i192", 4), ("tiny", 1000),
                                    ("qwen_decode", 1024), ("qwen_decode", 12),
                                    ("mixtral_decode", 16), ("tiny", 9)])
def test_layer_forward_equals_component_calls(name, T):
    """moe_layer_forward gives bit-identical results to moe_route ->
    moe_permute -> moe_grouped_ffn -> moe_combine on the same inputs (for
    T <= 8 the layer runs router, permutation and row gather as one launch;
    for T > 256 its top-k kernel also writes the permutation's bitmap)."""
    if name == "tiny_i192":   # no fused decode FFN (I_sub % 128 != 0): gate|up, down
        wl = replace(WL.TINY, I_sub=192, name="tiny-i192")
    else:
        wl = WL.ALL[name]
    wl = wl if T is None else wl.with_T(T)
    d = make_layer_inputs(wl, DEV)
    desc = B.desc_for(wl, expert_bias=d["expert_bias"])
    layer = B.MoeLayer(desc, DEV)
    out = layer.forward(d["x"], d["router_w"], d["w_gate_up"], d["w_down"], d["k_per_token"])
    assert layer.device_status() == 0
    Tt, k_max, E_r = wl.T, wl.k_max, wl.E_r
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx = torch.empty(Tt, k_max, dtype=torch.int32, device=DEV)
    w = torch.empty(Tt, k_max, dtype=torch.float32, device=DEV)
    counts = torch.empty(E_r, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E_r + 1, dtype=torch.int32, device=DEV)
    st_tok = torch.empty(Tt * k_max, dtype=torch.int32, device=DEV)
    inv = torch.empty(Tt * k_max, dtype=torch.int32, device=DEV)
    y = torch.empty(Tt * k_max, wl.H, dtype=torch.bfloat16, device=DEV)
    out2 = torch.empty(Tt, wl.H, dtype=torch.bfloat16, device=DEV)
    B.check(B.moe_route(desc, d["x"], d["router_w"], None, d["k_per_token"], None, idx, w, st, ws))
    B.check(B.moe_permute(desc, idx, d["k_per_token"], counts, offsets, st_tok, inv, st, ws))
    B.check(B.moe_grouped_ffn(desc, d["x"], st_tok, offsets, d["w_gate_up"], d["w_down"], y, st,
                              ws))
    B.check(B.moe_combine(desc, y, None, inv, w, d["k_per_token"], out2, st))
    assert B.moe_get_device_status(st) == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("mode", ["batch_max", "coarse"])
@pytest.mark.parametrize("name,T", [("tiny", None), ("qwen_decode", 64)])
def test_layer_comparison_budget_modes(name, T, mode):
    """The comparison modes run the same kernels on other budgets: every token
    at the batch maximum (uniform-k execution) or at whole experts
    n_sub * ceil(k / n_sub); the layer still matches the oracle."""
    from aware_moe_expert_gb300.inputs import apply_k_mode
    wl = WL.ALL[name] if T is None else WL.ALL[name].with_T(T)
    d = make_layer_inputs(wl, DEV)
    d["k_per_token"] = apply_k_mode(d["k_per_token"], mode, wl.n_sub, wl.k_max)
    desc = B.desc_for(wl, expert_bias=d["expert_bias"])
    layer = B.MoeLayer(desc, DEV)
    out = layer.forward(d["x"], d["router_w"], d["w_gate_up"], d["w_down"], d["k_per_token"])
    assert layer.device_status() == 0
    Lg = torch.empty(wl.T, wl.E_r, dtype=torch.float32, device=DEV)
    idx = torch.empty(wl.T, wl.k_max, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.k_max, dtype=torch.float32, device=DEV)
    B.check(B.moe_route(desc, d["x"], d["router_w"], None, d["k_per_token"], Lg, idx, w,
                        layer.status, layer.workspace))
    _compare(wl, d, desc, out, Lg, idx, np.arange(wl.T))


@pytest.mark.parametrize("path", [B.PATH_AUTO, B.PATH_PREFILL, B.PATH_DECODE])
def test_zero_tokens_is_a_no_op(path):
    """T = 0 through the layer and every component call: MOE_OK, no device
    error, nothing written."""
    wl = WL.TINY.with_T(1)
    d = make_layer_inputs(wl, DEV)
    desc = B.desc_for(wl, expert_bias=d["expert_bias"])
    desc.T = 0
    desc.path = path
    ws = torch.empty(max(B.moe_workspace_size(desc), 256), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    one_i = torch.zeros(1, dtype=torch.int32, device=DEV)
    one_f = torch.zeros(1, dtype=torch.float32, device=DEV)
    sentinel = torch.full((4, wl.H), 7.0, dtype=torch.bfloat16, device=DEV)
    B.check(B.moe_layer_forward(desc, sentinel, d["router_w"], d["w_gate_up"], d["w_down"],
                                one_i, sentinel, st, ws))
    B.check(B.moe_route(desc, sentinel, d["router_w"], None, one_i, None, one_i, one_f, st, ws))
    B.check(B.moe_permute(desc, one_i, one_i, one_i, one_i, one_i, one_i, st, ws))
    B.check(B.moe_combine(desc, sentinel, None, one_i, one_f, one_i, sentinel, st))
    assert B.moe_get_device_status(st) == 0
    assert bool((sentinel == 7.0).all())


@pytest.mark.parametrize("T", [129, 1000, 4097])
def test_layer_prefill_ragged_token_counts(T):
    """Token counts that leave partial 128-row router tiles and ragged unit
    tails on the prefill path (tensor-core router, gathering grouped GEMM);
    every token up to 1000, else a seeded sample plus the first and last."""
    wl = replace(WL.QWEN_DECODE, name="qwen-shape-prefill-ragged", phase="prefill", T=T)
    wl, d, desc, out, Lg, idx = _run_layer(wl, path=B.PATH_PREFILL)
    if T <= 1000:
        tokens = np.arange(T)
    else:
        rng = np.random.default_rng(T)
        tokens = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 256, replace=False)]))
    fro, n_tied = _compare(wl, d, desc, out, Lg, idx, tokens)
    assert fro <= 5e-3


@pytest.mark.gpu
@pytest.mark.parametrize("name,T", [("qwen_decode", 1), ("qwen_decode", 8), ("mixtral_decode", None),
                                    ("tiny", 300)])
def test_host_buffer_forward_matches_the_device_forward(name, T):
    """moe_layer_forward_host (x and k copied in from pinned host memory, out
    copied back) gives exactly what moe_layer_forward gives on device copies
    of the same inputs, on two calls in a row."""
    wl = WL.ALL[name] if T is None else WL.ALL[name].with_T(T)
    d = make_layer_inputs(wl, DEV)
    desc = B.desc_for(wl, expert_bias=d["expert_bias"])
    layer = B.MoeLayer(desc, DEV)
    ref = layer.forward(d["x"], d["router_w"], d["w_gate_up"], d["w_down"], d["k_per_token"])
    assert layer.device_status() == 0
    x_h = d["x"].cpu().pin_memory()
    k_h = d["k_per_token"].cpu().pin_memory()
    x_d = torch.empty_like(d["x"])
    k_d = torch.empty_like(d["k_per_token"])
    out_d = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):
        out_h = torch.zeros(wl.T, wl.H, dtype=torch.bfloat16).pin_memory()
        B.check(B.moe_layer_forward_host(desc, x_h, k_h, out_h, x_d, k_d, out_d, d["router_w"],
                                         d["w_gate_up"], d["w_down"], st, layer.workspace),
                "moe_layer_forward_host")
        assert B.moe_get_device_status(st) == 0     # synchronises the stream
        assert torch.equal(out_h.view(torch.int16), ref.cpu().view(torch.int16))
