"""GPU parity of routing (top-k_t and gates) and of the router logits.

Routing is bit-exact given the same fp32 logits: both sides receive logits
drawn by the seeded input generator.  Router logits from x and router_w are
compared with the oracle's float64 logits within an fp32 accumulation bound.
"""
import numpy as np
import pytest
import torch

from aware_moe_expert_gb300 import binding as B
from aware_moe_expert_gb300.inputs import make_logits, bf16_bits
from oracle import moe_oracle as O
from parity_utils import W_RTOL

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _route_given(desc, L, k):
    T, E_r, k_max = desc.T, desc.E_r, desc.k_max
    idx = torch.full((T, k_max), -7, dtype=torch.int32, device=DEV)
    w = torch.full((T, k_max), -7.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    B.check(B.moe_route(desc, None, None, L, k, None, idx, w, st, ws), "moe_route")
    code = B.moe_get_device_status(st)
    return idx.cpu().numpy(), w.cpu().numpy(), code


@pytest.mark.parametrize("E_r,k_max,T", [(32, 8, 64), (64, 8, 100), (128, 8, 513), (256, 16, 1024),
                                         (256, 32, 97), (7, 5, 33)])
@pytest.mark.parametrize("kind", ["normal", "ties", "flat"])
@pytest.mark.parametrize("score,renorm,scale", [("softmax", False, 1.0), ("softmax", True, 2.0),
                                                ("sigmoid", True, 1.0), ("sigmoid", False, 0.5)])
def test_topk_bit_exact_given_logits(E_r, k_max, T, kind, score, renorm, scale):
    L = make_logits(T, E_r, DEV, seed=E_r * 7 + T, kind=kind)
    g = torch.Generator().manual_seed(T)
    k = torch.randint(1, k_max + 1, (T,), generator=g, dtype=torch.int32).to(DEV)
    desc = B.LayerDesc(T=T, H=64, n_experts=E_r, n_sub=1, I_sub=64, k_max=k_max, score=score,
                       renorm=renorm, route_scale=scale)
    idx, w, code = _route_given(desc, L, k)
    assert code == 0, B.STATUS_NAMES[code]
    Ln = L.cpu().numpy()
    kn = k.cpu().numpy()
    want_idx, flags = O.select_topk(Ln, kn, k_max)
    assert flags == 0
    np.testing.assert_array_equal(idx, want_idx)
    want_w = O.gate_weights(Ln, want_idx, kn, score, renorm, scale)
    np.testing.assert_allclose(w, want_w, rtol=W_RTOL, atol=1e-30)


def test_topk_signed_zero_nan_and_k_range_flags():
    T, E_r, k_max = 8, 40, 6
    L = torch.zeros(T, E_r)
    L[0, 5] = -0.0
    L[0, 3] = 0.0
    L[1, :] = -0.0                       # all equal: lowest indices win
    L[2, 7] = float("nan")
    L[2, 9] = float("-inf")
    L[3, 11] = float("inf")
    L = L.to(DEV)
    k = torch.tensor([6, 6, 6, 6, 1, 2, 3, 4], dtype=torch.int32, device=DEV)
    desc = B.LayerDesc(T=T, H=64, n_experts=E_r, n_sub=1, I_sub=64, k_max=k_max)
    idx, w, code = _route_given(desc, L, k)
    assert code == 6  # MOE_ERR_NONFINITE
    want_idx, flags = O.select_topk(L.cpu().numpy(), k.cpu().numpy(), k_max)
    assert flags & O.FLAG_NONFINITE
    np.testing.assert_array_equal(idx, want_idx)
    # k out of range is reported and the row clamped
    L2 = make_logits(4, E_r, DEV, seed=3)
    k2 = torch.tensor([1, 0, 7, 2], dtype=torch.int32, device=DEV)
    idx2, _, code2 = _route_given(B.LayerDesc(T=4, H=64, n_experts=E_r, n_sub=1, I_sub=64,
                                              k_max=k_max), L2, k2)
    assert code2 == 7  # MOE_ERR_K_RANGE
    want2, flags2 = O.select_topk(L2.cpu().numpy(), k2.cpu().numpy(), k_max)
    assert flags2 & O.FLAG_K_RANGE
    np.testing.assert_array_equal(idx2, want2)


@pytest.mark.parametrize("T,H,n_experts,n_sub", [(64, 256, 16, 4), (64, 4096, 8, 4),
                                                 (200, 2048, 128, 1), (1024, 2048, 128, 2),
                                                 (300, 7168, 256, 1), (5, 512, 3, 3),
                                                 (1, 2048, 128, 2), (8, 7168, 256, 1),
                                                 (9, 2048, 128, 2), (127, 2048, 64, 2),
                                                 (130, 4096, 8, 4), (3, 12288, 16, 2),
                                                 (4, 16384, 4, 2), (17, 64, 1, 1)])
def test_router_logits_match_fp64(T, H, n_experts, n_sub):
    """Logits from the cluster router (CUDA cores, small T or other E_r), the
    sliced CUDA-core kernel (H > 12288) or the tensor-core GEMM."""
    g = torch.Generator(device=DEV).manual_seed(T + H)
    E_r = n_experts * n_sub
    x = torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16)
    rw = (torch.randn(E_r, H, generator=g, device=DEV) / H ** 0.5).to(torch.bfloat16)
    bias = torch.randn(n_experts, generator=g, device=DEV)
    k = torch.full((T,), 1, dtype=torch.int32, device=DEV)
    desc = B.LayerDesc(T=T, H=H, n_experts=n_experts, n_sub=n_sub, I_sub=64, k_max=1,
                       expert_bias=bias)
    L = torch.empty(T, E_r, dtype=torch.float32, device=DEV)
    idx = torch.empty(T, 1, dtype=torch.int32, device=DEV)
    w = torch.empty(T, 1, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    B.check(B.moe_route(desc, x, rw, None, k, L, idx, w, st, ws), "moe_route")
    assert B.moe_get_device_status(st) == 0
    X = O.bf16_to_f64(bf16_bits(x))
    R = O.bf16_to_f64(bf16_bits(rw))
    ref = O.router_logits(X, R, bias.cpu().numpy(), n_sub)
    # fp32 accumulation of exact bf16 products: |err| <= H * 2^-24 * sum|x w| (loose)
    mag = np.abs(X) @ np.abs(R).T
    err = np.abs(L.cpu().numpy().astype(np.float64) - ref)
    assert (err <= H * 2.0 ** -24 * mag + 1e-6).all(), f"max err {err.max():.3e}"


# From x through the tensor-core router with K split more than twice: softmax
# scores take the top-k kernel whose helper warps compute the softmax
# statistics while the selecting warps run, as long as its grid (T / 8 CTAs)
# fits one CTA per SM; (1216, 128) is the last such T on a 152-SM GB300 and
# (1224, 128) the first without.  Selection on the GPU's own fp32 logits is
# bit-exact, the gates within the fp32 bound.
@pytest.mark.parametrize("T,n_experts,n_sub,k_max", [(200, 64, 1, 8), (1024, 128, 2, 16),
                                                     (1216, 128, 1, 8), (1224, 128, 1, 8)])
@pytest.mark.parametrize("renorm,scale", [(False, 1.0), (True, 2.5)])
def test_split_k_router_top_k_on_its_own_logits(T, n_experts, n_sub, k_max, renorm, scale):
    H = 2048
    E_r = n_experts * n_sub
    g = torch.Generator(device=DEV).manual_seed(T + E_r)
    x = torch.randn(T, H, generator=g, device=DEV).to(torch.bfloat16)
    rw = (torch.randn(E_r, H, generator=g, device=DEV) / H ** 0.5).to(torch.bfloat16)
    bias = torch.randn(n_experts, generator=g, device=DEV) * 0.1
    k = torch.randint(1, k_max + 1, (T,), generator=torch.Generator().manual_seed(T),
                      dtype=torch.int32).to(DEV)
    desc = B.LayerDesc(T=T, H=H, n_experts=n_experts, n_sub=n_sub, I_sub=64, k_max=k_max,
                       score="softmax", renorm=renorm, route_scale=scale, expert_bias=bias)
    L = torch.empty(T, E_r, dtype=torch.float32, device=DEV)
    idx = torch.full((T, k_max), -7, dtype=torch.int32, device=DEV)
    w = torch.full((T, k_max), -7.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    B.check(B.moe_route(desc, x, rw, None, k, L, idx, w, st, ws), "moe_route")
    assert B.moe_get_device_status(st) == 0
    Ln, kn = L.cpu().numpy(), k.cpu().numpy()
    want_idx, flags = O.select_topk(Ln, kn, k_max)
    assert flags == 0
    np.testing.assert_array_equal(idx.cpu().numpy(), want_idx)
    want_w = O.gate_weights(Ln, want_idx, kn, "softmax", renorm, scale)
    np.testing.assert_allclose(w.cpu().numpy(), want_w, rtol=W_RTOL, atol=1e-30)
