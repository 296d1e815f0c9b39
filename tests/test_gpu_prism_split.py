"""MoE-Prism's split, end to end on the GPU (arXiv 2510.19366, §III-B1 Eq. (3)
and §III-B2): an expert's intermediate neurons cut into n_sub slices give
n_sub sub-experts whose outputs add up to the expert's.  With the linear gate
initialised by repeating each expert's router row n_sub times, k = n_sub *
k_orig and route_scale = n_sub, the split layer selects exactly the
sub-experts of the top-k_orig experts with gate p_e / n_sub * n_sub = p_e, so
it reproduces the unsplit layer.  Both layers run through moe_layer_forward
on the same x; their outputs must agree within the layer tolerance (they
differ only by the bf16 rounding of act and y in different places), and the
unsplit one must match the oracle.
"""
import math

import numpy as np
import pytest
import torch

from aware_moe_expert_gb300 import binding as B
from oracle import moe_oracle as O
from aware_moe_expert_gb300.inputs import bf16_bits
from parity_utils import assert_close_layer, spec_of, unit_fetch

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _split_weights(wgu, wd, n_sub):
    """[E, 2I, H], [E, H, I] -> [E n_sub, 2 I/n, H], [E n_sub, H, I/n] (contiguous slices)."""
    E, two_i, H = wgu.shape
    I = two_i // 2
    Is = I // n_sub
    gate = wgu[:, :I, :].reshape(E, n_sub, Is, H)
    up = wgu[:, I:, :].reshape(E, n_sub, Is, H)
    wgu_s = torch.cat([gate, up], dim=2).reshape(E * n_sub, 2 * Is, H).contiguous()
    wd_s = wd.reshape(E, H, n_sub, Is).permute(0, 2, 1, 3).reshape(E * n_sub, H, Is).contiguous()
    return wgu_s, wd_s


@pytest.mark.parametrize("T", [8, 64, 300])
def test_split_layer_reproduces_unsplit_layer(T):
    E, H, I, n_sub, k_orig = 8, 256, 512, 4, 2
    g = torch.Generator(device=DEV).manual_seed(77)
    x = torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16)
    wgu = (torch.randn(E, 2 * I, H, generator=g, device=DEV) / math.sqrt(H)).to(torch.bfloat16)
    wd = (torch.randn(E, H, I, generator=g, device=DEV) / math.sqrt(I)).to(torch.bfloat16)
    rw = (torch.randn(E, H, generator=g, device=DEV) / math.sqrt(H)).to(torch.bfloat16)
    k_u = torch.full((T,), k_orig, dtype=torch.int32, device=DEV)
    k_s = torch.full((T,), k_orig * n_sub, dtype=torch.int32, device=DEV)

    desc_u = B.LayerDesc(T=T, H=H, n_experts=E, n_sub=1, I_sub=I, k_max=k_orig)
    out_u = B.MoeLayer(desc_u, DEV)
    y_u = out_u.forward(x, rw, wgu, wd, k_u)
    assert out_u.device_status() == 0

    wgu_s, wd_s = _split_weights(wgu, wd, n_sub)
    rw_s = rw.repeat_interleave(n_sub, dim=0).contiguous()   # unit e*n_sub + n gets row e
    desc_s = B.LayerDesc(T=T, H=H, n_experts=E, n_sub=n_sub, I_sub=I // n_sub,
                         k_max=k_orig * n_sub, route_scale=float(n_sub))
    out_s = B.MoeLayer(desc_s, DEV)
    y_s = out_s.forward(x, rw_s, wgu_s, wd_s, k_s)
    assert out_s.device_status() == 0

    # the split layer selected exactly the sub-experts of the experts the
    # unsplit layer selected
    idx_u = torch.empty(T, k_orig, dtype=torch.int32, device=DEV)
    idx_s = torch.empty(T, k_orig * n_sub, dtype=torch.int32, device=DEV)
    w_u = torch.empty(T, k_orig, dtype=torch.float32, device=DEV)
    w_s = torch.empty(T, k_orig * n_sub, dtype=torch.float32, device=DEV)
    L_u = torch.empty(T, E, dtype=torch.float32, device=DEV)
    B.check(B.moe_route(desc_u, x, rw, None, k_u, L_u, idx_u, w_u, out_u.status, out_u.workspace))
    B.check(B.moe_route(desc_s, x, rw_s, None, k_s, None, idx_s, w_s, out_s.status,
                        out_s.workspace))
    eu = idx_u.cpu().numpy()
    es = idx_s.cpu().numpy() // n_sub
    for t in range(T):
        assert sorted(set(es[t].tolist())) == sorted(eu[t].tolist())
    # each selected sub-expert carries its expert's gate (p_e / n_sub * n_sub)
    wu, ws = w_u.cpu().numpy(), w_s.cpu().numpy()
    for t in range(T):
        ref = dict(zip(eu[t].tolist(), wu[t].tolist()))
        for u, w in zip(idx_s.cpu().numpy()[t].tolist(), ws[t].tolist()):
            assert abs(w - ref[u // n_sub]) <= 2e-5 * abs(ref[u // n_sub])

    assert_close_layer(y_s.double().cpu().numpy(), y_u.double().cpu().numpy(), "split vs unsplit")
    # and the unsplit layer against the oracle (routed from the GPU's fp32
    # logits, so that a near tie cannot select differently)
    spec = spec_of(desc_u)
    ref = O.layer_forward(spec, bf16_bits(x), None, unit_fetch(wgu), unit_fetch(wd),
                          k_u.cpu().numpy(), logits=L_u.cpu().numpy())
    assert_close_layer(y_u.double().cpu().numpy(), ref["out"], "unsplit vs oracle")
