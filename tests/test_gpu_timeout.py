"""Bounded device waits: a test-only flag makes the FFN producer skip its
first load, so the consumer's wait on that ring slot must give up (about two
seconds), report MOE_ERR_DEVICE_TIMEOUT in the status word, drain and return.
The context stays usable: a normal call right after matches the oracle."""
import math

import numpy as np
import pytest
import torch

from aware_moe_expert_gb300 import binding as B
from aware_moe_expert_gb300.inputs import make_logits, bf16_bits
from oracle import moe_oracle as O
from parity_utils import assert_close_layer, spec_of, unit_fetch

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _setup(path, debug):
    T, H, n_experts, n_sub, I_sub, k_max = 64, 256, 16, 4, 128, 8
    E_r = n_experts * n_sub
    g = torch.Generator(device=DEV).manual_seed(5)
    x = torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16)
    wgu = (torch.randn(E_r, 2 * I_sub, H, generator=g, device=DEV) / math.sqrt(H)).to(torch.bfloat16)
    wd = (torch.randn(E_r, H, I_sub, generator=g, device=DEV) / math.sqrt(512)).to(torch.bfloat16)
    L = make_logits(T, E_r, DEV, seed=11)
    k = torch.randint(1, k_max + 1, (T,), generator=torch.Generator().manual_seed(3),
                      dtype=torch.int32).to(DEV)
    desc = B.LayerDesc(T=T, H=H, n_experts=n_experts, n_sub=n_sub, I_sub=I_sub, k_max=k_max,
                       path=path, debug_flags=debug)
    return desc, x, wgu, wd, L, k


def _ffn(desc, x, wgu, wd, L, k):
    T, k_max, E_r = desc.T, desc.k_max, desc.E_r
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx = torch.empty(T, k_max, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k_max, dtype=torch.float32, device=DEV)
    counts = torch.empty(E_r, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E_r + 1, dtype=torch.int32, device=DEV)
    st_tok = torch.empty(T * k_max, dtype=torch.int32, device=DEV)
    inv = torch.empty(T * k_max, dtype=torch.int32, device=DEV)
    y = torch.zeros(T * k_max, desc.H, dtype=torch.bfloat16, device=DEV)
    B.check(B.moe_route(desc, None, None, L, k, None, idx, w, st, ws))
    B.check(B.moe_permute(desc, idx, k, counts, offsets, st_tok, inv, st, ws))
    assert B.moe_get_device_status(st) == 0
    B.check(B.moe_grouped_ffn(desc, x, st_tok, offsets, wgu, wd, y, st, ws))
    return B.moe_get_device_status(st), y


@pytest.mark.parametrize("path", [B.PATH_PREFILL, B.PATH_DECODE, "pair"])
def test_skipped_load_times_out_and_context_survives(path):
    extra = 0
    if path == "pair":                     # the CTA-pair GEMM's leader skips the load
        path, extra = B.PATH_PREFILL, B.DEBUG_FORCE_PAIR
    desc, x, wgu, wd, L, k = _setup(path, B.DEBUG_SKIP_FIRST_LOAD | extra)
    code, _ = _ffn(desc, x, wgu, wd, L, k)
    assert code == 5, B.STATUS_NAMES.get(code, code)     # MOE_ERR_DEVICE_TIMEOUT
    # the same context keeps working (same kernel family)
    desc.debug_flags = extra
    code, y = _ffn(desc, x, wgu, wd, L, k)
    assert code == 0
    ref = O.layer_forward(spec_of(desc), bf16_bits(x), None, unit_fetch(wgu), unit_fetch(wd),
                          k.cpu().numpy(), logits=L.cpu().numpy())
    assert_close_layer(y[: ref["n_assign"]].to(torch.float64).cpu().numpy(), ref["y_perm"])


def test_layer_forward_gathering_ffn_times_out_and_context_survives():
    """The same through moe_layer_forward, whose fused decode FFN gathers its
    token rows itself (four more warps on the stage barriers): the skipped
    load must still end every wait, and a normal call afterwards is right."""
    desc, x, wgu, wd, L, k = _setup(B.PATH_DECODE, B.DEBUG_SKIP_FIRST_LOAD)
    g = torch.Generator(device=DEV).manual_seed(9)
    router_w = (torch.randn(desc.E_r, desc.H, generator=g, device=DEV)
                / math.sqrt(desc.H)).to(torch.bfloat16)
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty(desc.T, desc.H, dtype=torch.bfloat16, device=DEV)
    B.check(B.moe_layer_forward(desc, x, router_w, wgu, wd, k, out, st, ws))
    assert B.moe_get_device_status(st) == 5                    # MOE_ERR_DEVICE_TIMEOUT
    desc.debug_flags = 0
    st.zero_()
    B.check(B.moe_layer_forward(desc, x, router_w, wgu, wd, k, out, st, ws))
    assert B.moe_get_device_status(st) == 0
    ref = O.layer_forward(spec_of(desc), bf16_bits(x), bf16_bits(router_w), unit_fetch(wgu),
                          unit_fetch(wd), k.cpu().numpy())
    got = out.to(torch.float64).cpu().numpy()
    # fp32 GPU logits vs fp64 oracle logits: compare tokens away from near ties
    from parity_utils import tie_safe_tokens
    Lg = torch.empty(desc.T, desc.E_r, dtype=torch.float32, device=DEV)
    idx = torch.empty(desc.T, desc.k_max, dtype=torch.int32, device=DEV)
    w = torch.empty(desc.T, desc.k_max, dtype=torch.float32, device=DEV)
    B.check(B.moe_route(desc, x, router_w, None, k, Lg, idx, w, st, ws))
    L64 = ref["logits"]
    delta = 2.0 * np.abs(Lg.cpu().numpy().astype(np.float64) - L64).max(axis=1) + 1e-7
    ok, n_tied = tie_safe_tokens(L64, idx.cpu().numpy(), k.cpu().numpy(), delta)
    assert n_tied <= 2
    assert_close_layer(got[ok], ref["out"][ok], "out")
