"""GPU parity of the grouped SwiGLU FFN (gate|up with fused SiLU*mul, then
down) and of the shared expert, row by row against the fp64 oracle.

Routing comes from logits drawn by the input generator and given to both
sides, so both run the same permutation; shapes span several 128-row tiles
per unit with ragged tails, empty units, and every tile-width variant of the
kernels (I_sub multiple of 128 or only of 64; H multiple of 256, 128 or 64).
"""
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


def _weights(E_r, H, I_sub, n_sub, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    wgu = (torch.randn(E_r, 2 * I_sub, H, generator=g, device=DEV) / math.sqrt(H)).to(torch.bfloat16)
    wd = (torch.randn(E_r, H, I_sub, generator=g, device=DEV)
          / math.sqrt(n_sub * I_sub)).to(torch.bfloat16)
    x = torch.randn(4096, H, generator=g, device=DEV).to(torch.bfloat16)
    return x, wgu, wd


@pytest.mark.parametrize("path", [B.PATH_PREFILL, B.PATH_DECODE, "pair"])
@pytest.mark.parametrize("T,H,n_experts,n_sub,I_sub,k_max,skew", [
    (64, 256, 16, 4, 128, 8, 0.0),      # tiny layer shape
    (300, 512, 8, 1, 192, 4, 3.0),      # 3 m-tiles on hot units, I_sub % 128 != 0
    (257, 384, 4, 2, 256, 3, 0.0),      # H % 256 != 0 (down uses 128-wide tiles)
    (130, 320, 6, 1, 64, 2, 6.0),       # H % 128 != 0 (64-wide tiles), empty units
    (1, 2048, 128, 2, 384, 16, 0.0),    # one token (decode: split-K over few items)
    (8, 2048, 128, 2, 384, 16, 0.0),    # eight tokens
    (400, 512, 4, 2, 256, 4, 4.0),      # > 128 rows on a unit: decode chunks of 128 tokens
    (1500, 256, 8, 1, 128, 4, 1.5),     # units of hundreds of rows: 256-row pair tiles + tails
    (2000, 256, 16, 1, 128, 6, 0.7),    # remainders on both sides of 128 rows
])
def test_grouped_ffn_rows_match_oracle(T, H, n_experts, n_sub, I_sub, k_max, skew, path):
    """Every kernel family (prefill tiles on one CTA or on CTA pairs with
    256-row and 128-row tiles, decode swap-AB) on the same inputs; shapes a
    family does not support fall back to another one."""
    debug = 0
    if path == "pair":
        path, debug = B.PATH_PREFILL, B.DEBUG_FORCE_PAIR
    E_r = n_experts * n_sub
    x, wgu, wd = _weights(E_r, H, I_sub, n_sub, seed=T * 31 + H)
    x = x[:T].contiguous()
    L = make_logits(T, E_r, DEV, seed=T + E_r)
    if skew:
        L = L + (-skew * torch.log(torch.arange(1, E_r + 1, device=DEV, dtype=torch.float32)))
    g = torch.Generator().manual_seed(T)
    k = torch.randint(1, k_max + 1, (T,), generator=g, dtype=torch.int32).to(DEV)
    desc = B.LayerDesc(T=T, H=H, n_experts=n_experts, n_sub=n_sub, I_sub=I_sub, k_max=k_max,
                       path=path, debug_flags=debug)
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx = torch.empty(T, k_max, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k_max, dtype=torch.float32, device=DEV)
    counts = torch.empty(E_r, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E_r + 1, dtype=torch.int32, device=DEV)
    st_tok = torch.empty(T * k_max, dtype=torch.int32, device=DEV)
    inv = torch.empty(T * k_max, dtype=torch.int32, device=DEV)
    y = torch.zeros(T * k_max, H, dtype=torch.bfloat16, device=DEV)
    B.check(B.moe_route(desc, None, None, L, k, None, idx, w, st, ws))
    B.check(B.moe_permute(desc, idx, k, counts, offsets, st_tok, inv, st, ws))
    B.check(B.moe_grouped_ffn(desc, x, st_tok, offsets, wgu, wd, y, st, ws))
    assert B.moe_get_device_status(st) == 0
    ref = O.layer_forward(spec_of(desc), bf16_bits(x), None, unit_fetch(wgu), unit_fetch(wd),
                          k.cpu().numpy(), logits=L.cpu().numpy())
    n = ref["n_assign"]
    np.testing.assert_array_equal(offsets.cpu().numpy(), ref["offsets"])
    got = y[:n].to(torch.float64).cpu().numpy()
    assert_close_layer(got, ref["y_perm"], "y_perm")


@pytest.mark.parametrize("T,H,I_sh", [
    (100, 256, 128), (300, 512, 192),   # one-CTA tiles
    (700, 512, 256), (1024, 256, 128),  # CTA pairs (ragged last pair tile; exact)
])
def test_shared_expert_matches_oracle(T, H, I_sh):
    g = torch.Generator(device=DEV).manual_seed(T)
    x = torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16)
    sgu = (torch.randn(2 * I_sh, H, generator=g, device=DEV) / math.sqrt(H)).to(torch.bfloat16)
    sd = (torch.randn(H, I_sh, generator=g, device=DEV) / math.sqrt(I_sh)).to(torch.bfloat16)
    desc = B.LayerDesc(T=T, H=H, n_experts=4, n_sub=1, I_sub=64, k_max=2, I_shared=I_sh,
                       w_shared_gate_up=sgu, w_shared_down=sd)
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    B.check(B.moe_shared_ffn(desc, x, y, st, ws))
    assert B.moe_get_device_status(st) == 0
    ref = O.swiglu_ffn(O.bf16_to_f64(bf16_bits(x)), O.bf16_to_f64(bf16_bits(sgu)),
                       O.bf16_to_f64(bf16_bits(sd)))
    assert_close_layer(y.to(torch.float64).cpu().numpy(), ref, "y_shared")
