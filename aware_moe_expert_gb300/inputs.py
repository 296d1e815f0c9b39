"""Seeded synthetic inputs for the MoE layer (shared by the CUDA path's tests,
the bench and the oracle's tests).

This module holds no arithmetic of the layer: it only draws numbers.  Every
tensor has its own torch generator seeded from (workload seed, tensor id), so
a tensor does not change when another one is added or resized.  Normal draws
are made in float32 and rounded to bf16 (round to nearest even, torch's
conversion); the same bits then feed both the CUDA library and the oracle.

Distributions:
  x                 ~ N(0, 1)
  router_w          ~ N(0, 1/H), or N(0, router_std^2) when given
  w_gate_up (gate and up rows)   ~ N(0, 1/H)       (fan_in = H)
  w_down            ~ N(0, 1/I)  with I = n_sub * I_sub, the intermediate size
                      of the monolithic expert the sub-experts slice (fan_in)
  shared expert     the same rules with I = I_shared
  expert bias       N(0, 1) per expert, or -s * ln(rank) with a seeded random
                    rank permutation (Zipf(s) popularity in logit space)
  k_per_token       uniform over the workload's choices, drawn per token or per
                    request (then shared by the request's tokens)
  proxy router      expert-level router_w_expert ~ N(0, 1/H) (or router_std);
                    gate neurons: r distinct local indices per unit, uniformly
                    at random (a stand-in for the co-activation calibration,
                    which needs real activations); allocation table: k split as
                    evenly as possible over the m kept experts, the
                    higher-ranked ones taking the remainder
"""
from __future__ import annotations

import math
from typing import Dict, Optional

import torch

from .workloads import Workload

_IDS = {"x": 1, "router_w": 2, "w_gate_up": 3, "w_down": 4, "bias": 5, "k": 6,
        "w_shared_gate_up": 7, "w_shared_down": 8, "logits": 9, "router_w_expert": 10,
        "gate_neurons": 11}


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000 + _IDS[name])
    return g


def _normal_bf16(shape, std: float, g: torch.Generator, device, chunk_dim0: bool = True):
    """N(0, std^2) draws rounded to bf16, generated in slabs along dim 0 to
    bound the float32 temporary."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if len(shape) >= 3 and chunk_dim0:
        for i in range(shape[0]):
            out[i] = (torch.randn(shape[1:], generator=g, device=device,
                                  dtype=torch.float32) * std).to(torch.bfloat16)
    else:
        out.copy_((torch.randn(shape, generator=g, device=device, dtype=torch.float32)
                   * std).to(torch.bfloat16))
    return out


def draw_k(wl: Workload, device="cpu", seed: Optional[int] = None) -> torch.Tensor:
    seed = wl.seed if seed is None else seed
    g = _gen(seed, "k", "cpu")
    choices = torch.tensor(wl.k_choices, dtype=torch.int32)
    if wl.k_per == "token":
        pick = torch.randint(0, len(choices), (wl.T,), generator=g)
        k = choices[pick]
    else:
        n_req = (wl.T + wl.tokens_per_request - 1) // wl.tokens_per_request
        pick = torch.randint(0, len(choices), (n_req,), generator=g)
        k = choices[pick].repeat_interleave(wl.tokens_per_request)[: wl.T]
    return k.to(torch.int32).contiguous().to(device)


def draw_k_normal(T: int, mu: float, sigma: float, k_max: int, seed: int = 7,
                  device="cpu") -> torch.Tensor:
    """Budgets k = clip(round(x), 1, k_max), x ~ N(mu, sigma^2), one draw per
    token: the k-target generator of MoE-Prism §IV-B2, Eq. (7)."""
    g = torch.Generator().manual_seed(seed)
    x = mu + sigma * torch.randn(T, generator=g, dtype=torch.float64)
    return torch.round(x).clamp_(1, k_max).to(torch.int32).contiguous().to(device)


def apply_k_mode(k: torch.Tensor, mode: str, n_sub: int, k_max: int) -> torch.Tensor:
    """Budgets actually executed in a comparison mode:
    "exact" every token its own k; "batch_max" every token the batch maximum
    (what a uniform-k grouped kernel runs, MoE-Prism §III-C1); "coarse"
    n_sub * ceil(k / n_sub) (whole experts, MoE-Prism §V-D1), at most k_max."""
    if mode == "exact":
        return k
    if mode == "batch_max":
        return torch.full_like(k, int(k.max().item()))
    if mode == "coarse":
        return torch.clamp(((k + n_sub - 1) // n_sub) * n_sub, max=k_max).to(k.dtype)
    raise ValueError(f"unknown k mode {mode!r}")


def draw_bias(wl: Workload, seed: Optional[int] = None) -> Optional[torch.Tensor]:
    seed = wl.seed if seed is None else seed
    g = _gen(seed, "bias", "cpu")
    if wl.bias == "none":
        return None
    if wl.bias == "normal":
        return torch.randn(wl.n_experts, generator=g, dtype=torch.float32)
    if wl.bias == "zipf":
        rank = torch.randperm(wl.n_experts, generator=g).to(torch.float64) + 1.0
        return (-wl.zipf_s * torch.log(rank)).to(torch.float32)
    raise ValueError(wl.bias)


def make_layer_inputs(wl: Workload, device="cpu", seed: Optional[int] = None,
                      with_weights: bool = True) -> Dict[str, torch.Tensor]:
    """All inputs of one layer call, on ``device``.

    Keys: x [T,H] bf16, router_w [E_r,H] bf16, expert_bias [n_experts] f32 or
    None, w_gate_up [E_r, 2*I_sub, H] bf16, w_down [E_r, H, I_sub] bf16,
    k_per_token [T] int32, and for a shared expert w_shared_gate_up
    [2*I_shared, H] / w_shared_down [H, I_shared].
    """
    seed = wl.seed if seed is None else seed
    dev = torch.device(device)
    T, H, E_r, I_sub = wl.T, wl.H, wl.E_r, wl.I_sub
    d: Dict[str, torch.Tensor] = {}
    d["x"] = _normal_bf16((T, H), 1.0, _gen(seed, "x", dev), dev)
    rstd = wl.router_std if wl.router_std is not None else 1.0 / math.sqrt(H)
    d["router_w"] = _normal_bf16((E_r, H), rstd, _gen(seed, "router_w", dev), dev)
    b = draw_bias(wl, seed)
    d["expert_bias"] = None if b is None else b.to(dev)
    d["k_per_token"] = draw_k(wl, dev, seed)
    if with_weights:
        d["w_gate_up"] = _normal_bf16((E_r, 2 * I_sub, H), 1.0 / math.sqrt(H),
                                      _gen(seed, "w_gate_up", dev), dev)
        d["w_down"] = _normal_bf16((E_r, H, I_sub), 1.0 / math.sqrt(wl.I),
                                   _gen(seed, "w_down", dev), dev)
        if wl.I_shared > 0:
            d["w_shared_gate_up"] = _normal_bf16((2 * wl.I_shared, H), 1.0 / math.sqrt(H),
                                                 _gen(seed, "w_shared_gate_up", dev), dev)
            d["w_shared_down"] = _normal_bf16((H, wl.I_shared), 1.0 / math.sqrt(wl.I_shared),
                                              _gen(seed, "w_shared_down", dev), dev)
    return d


def draw_gate_neurons(wl: Workload, r: int, seed: Optional[int] = None) -> torch.Tensor:
    """int32 [E_r, r]: r distinct local neuron indices per unit (random)."""
    seed = wl.seed if seed is None else seed
    g = _gen(seed, "gate_neurons", "cpu")
    rows = [torch.randperm(wl.I_sub, generator=g)[:r] for _ in range(wl.E_r)]
    return torch.stack(rows).to(torch.int32)


def allocation_table(k_max: int, m: int, n_sub: int) -> torch.Tensor:
    """int32 [k_max + 1, m]: row k gives each of the m kept experts
    floor(k / m) sub-experts, plus one for the first k mod m of them."""
    rows = []
    for k in range(k_max + 1):
        rows.append([k // m + (1 if j < k % m else 0) for j in range(m)])
    t = torch.tensor(rows, dtype=torch.int32)
    if int(t.max()) > n_sub:
        raise ValueError("k_max exceeds m * n_sub")
    return t


def make_cg_inputs(wl: Workload, device="cpu", seed: Optional[int] = None, r: int = 8):
    """Inputs of the proxy router: router_w_expert bf16 [n_experts, H], gate
    neurons int32 [E_r, r], allocation table int32 [k_max + 1, native_m]."""
    seed = wl.seed if seed is None else seed
    dev = torch.device(device)
    rstd = wl.router_std if wl.router_std is not None else 1.0 / math.sqrt(wl.H)
    return {"router_w_expert": _normal_bf16((wl.n_experts, wl.H), rstd,
                                            _gen(seed, "router_w_expert", dev), dev),
            "gate_neurons": draw_gate_neurons(wl, r, seed).to(dev),
            "kappa": allocation_table(wl.k_max, wl.native_m, wl.n_sub).to(dev)}


def make_fold_tables(E_r: int, device="cpu", seed: int = 11):
    """Synthetic calibration tables for decode expert-pool folding (the pages'
    tables come from calibration data, out of scope here): S [E_r, E_r] scalar
    projectors ~ N(1, 0.25^2) clipped to [-4, 4] with S[u, u] = 1, and L
    [E_r, E_r] projection losses ~ U(0, 1) with L[u, u] = 0; fp32."""
    g = torch.Generator().manual_seed(seed)
    S = (1.0 + 0.25 * torch.randn(E_r, E_r, generator=g)).clamp_(-4.0, 4.0)
    S.fill_diagonal_(1.0)
    L = torch.rand(E_r, E_r, generator=g)
    L.fill_diagonal_(0.0)
    return S.float().contiguous().to(device), L.float().contiguous().to(device)


def make_paths(topk_idx: torch.Tensor, topk_w: torch.Tensor, mode: str = "share_source"):
    """Synthetic composed paths from a routing (a path router is trained, out
    of scope).  A token's selected units in slot order, u_0, u_1, ...; the
    path weight is the slot's gate weight.  Recipes:
      share_source   slot j targets u_j; even slots are their own source, odd
                     slots take u_{j-1} as source (consecutive paths share
                     an expansion)
      share_target   even slots are diagonal (u_j, u_j); odd slots keep u_j
                     as source and take u_{j-1} as target (consecutive paths
                     share a projection)
      duplicate      like share_target, and every slot j = 3 mod 4 repeats
                     the path of slot j - 1 (the same (source, target) twice)
    Returns (src_idx, tgt_idx, beta), -1 / 0 after k_t (slots past k_t are -1
    in topk_idx)."""
    k_max = topk_idx.shape[1]
    prev = topk_idx.clone()
    n_odd = k_max // 2
    prev[:, 1:2 * n_odd:2] = topk_idx[:, 0:2 * n_odd - 1:2]
    if mode == "share_source":
        src, tgt = prev, topk_idx.clone()
    elif mode in ("share_target", "duplicate"):
        src, tgt = topk_idx.clone(), prev
        if mode == "duplicate":
            src[:, 3::4] = src[:, 2:k_max - 1:4][:, :src[:, 3::4].shape[1]]
            tgt[:, 3::4] = tgt[:, 2:k_max - 1:4][:, :tgt[:, 3::4].shape[1]]
    else:
        raise ValueError(mode)
    live = topk_idx >= 0
    src = torch.where(live, src, torch.full_like(src, -1))
    tgt = torch.where(live, tgt, torch.full_like(tgt, -1))
    beta = torch.where(live, topk_w, torch.zeros_like(topk_w))
    return src.contiguous(), tgt.contiguous(), beta.contiguous()


def make_logits(T: int, E_r: int, device="cpu", seed: int = 7, kind: str = "normal"):
    """Float32 logits for routing-only tests.

    kind: "normal" N(0,1); "ties" values from a 5-point set so that many ties
    occur, with -0.0 and +0.0 both present; "flat" every logit equal.
    """
    g = _gen(seed, "logits", "cpu")
    if kind == "normal":
        L = torch.randn(T, E_r, generator=g, dtype=torch.float32)
    elif kind == "ties":
        vals = torch.tensor([-1.5, -0.0, 0.0, 0.25, 2.0], dtype=torch.float32)
        L = vals[torch.randint(0, len(vals), (T, E_r), generator=g)]
    elif kind == "flat":
        L = torch.full((T, E_r), 0.5, dtype=torch.float32)
    else:
        raise ValueError(kind)
    return L.contiguous().to(device)


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a bf16 tensor's bit patterns (for the oracle)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")
