"""GPU parity of decode expert-pool folding (moe_fold_decode,
moe_layer_forward_fold) against the CPU oracle (oracle/exfold.py).

The fold is integer and fp32 routing metadata: pool, targets, new budgets and
merged weights must equal the oracle's bit for bit (both sides add the same
fp32 numbers in the same order).  The folded layer's output is compared, in
the stated layer tolerance, with the fp64 oracle FFN over the folded routing
of the GPU's own route.
"""
import numpy as np
import pytest
import torch

from aware_moe_expert_gb300 import binding as B
from aware_moe_expert_gb300 import workloads as WL
from aware_moe_expert_gb300.inputs import make_fold_tables, make_layer_inputs, bf16_bits
from oracle import exfold as F
from oracle import moe_oracle as O
from parity_utils import assert_close_layer, unit_fetch

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _routing(T, E_r, k_max, seed, skew=0.0):
    g = torch.Generator().manual_seed(seed)
    k = torch.randint(1, k_max + 1, (T,), generator=g, dtype=torch.int32)
    idx = torch.full((T, k_max), -1, dtype=torch.int32)
    w = torch.zeros(T, k_max)
    pref = torch.exp(-skew * torch.arange(E_r, dtype=torch.float32) / E_r)
    for t in range(T):
        sel = torch.multinomial(pref, int(k[t]), replacement=False, generator=g)
        idx[t, :k[t]] = sel.to(torch.int32)
        w[t, :k[t]] = torch.rand(int(k[t]), generator=g)
    return idx, w, k


def _run_fold(desc, fold, idx, w, k):
    T, k_max = idx.shape
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    oi = torch.empty(T, k_max, dtype=torch.int32, device=DEV)
    ow = torch.empty(T, k_max, dtype=torch.float32, device=DEV)
    ok = torch.empty(T, dtype=torch.int32, device=DEV)
    pool = torch.empty(fold.D, dtype=torch.int32, device=DEV)
    B.check(B.moe_fold_decode(desc, fold, idx.to(DEV), w.to(DEV), k.to(DEV), oi, ow, ok, pool, st,
                              ws), "moe_fold_decode")
    return oi.cpu().numpy(), ow.cpu().numpy(), ok.cpu().numpy(), pool.cpu().numpy(), \
        B.moe_get_device_status(st)


@pytest.mark.parametrize("T,E_r,k_max,D,skew", [
    (1, 32, 8, 4, 0.0), (8, 256, 16, 16, 0.0), (64, 256, 16, 64, 2.0), (100, 64, 8, 8, 3.0),
    (1024, 256, 16, 96, 1.0), (65, 32, 8, 1, 0.0), (37, 48, 6, 48, 0.0)])
@pytest.mark.parametrize("static", [False, True])
def test_fold_bit_exact(T, E_r, k_max, D, skew, static):
    """Pool, targets, budgets and merged weights equal the oracle's exactly,
    for a dynamic pool and for a static one."""
    idx, w, k = _routing(T, E_r, k_max, seed=T * 7 + E_r, skew=skew)
    S, L = make_fold_tables(E_r, seed=E_r + D)
    pool_in = None
    if static:
        pool_in = torch.randperm(E_r, generator=torch.Generator().manual_seed(D))[:D].to(torch.int32)
    desc = B.LayerDesc(T=T, H=64, n_experts=E_r, n_sub=1, I_sub=64, k_max=k_max)
    fold = B.FoldDesc(D=D, S=S.to(DEV), L=L.to(DEV),
                      pool=None if pool_in is None else pool_in.to(DEV))
    oi, ow, ok, pool, code = _run_fold(desc, fold, idx, w, k)
    assert code == 0, B.STATUS_NAMES[code]
    wi, ww, wk, wpool = F.fold_decode(idx.numpy(), w.numpy(), k.numpy(), E_r, D, S.numpy(),
                                      L.numpy(), pool=None if pool_in is None else pool_in.numpy())
    np.testing.assert_array_equal(pool[:len(wpool)], wpool)
    np.testing.assert_array_equal(ok, wk)
    np.testing.assert_array_equal(oi, wi)
    np.testing.assert_array_equal(ow.view(np.uint32), ww.astype(np.float32).view(np.uint32))


def test_fold_reports_bad_static_pool():
    idx, w, k = _routing(16, 32, 4, seed=3)
    S, L = make_fold_tables(32)
    desc = B.LayerDesc(T=16, H=64, n_experts=32, n_sub=1, I_sub=64, k_max=4)
    fold = B.FoldDesc(D=3, S=S.to(DEV), L=L.to(DEV),
                      pool=torch.tensor([5, 5, 9], dtype=torch.int32, device=DEV))
    *_, code = _run_fold(desc, fold, idx, w, k)
    assert code == 8   # MOE_ERR_BAD_INDEX


@pytest.mark.parametrize("name,T,D", [("qwen_decode", 8, 24), ("qwen_decode", 64, 64),
                                      ("mixtral_decode", None, 12), ("tiny", None, 10)])
def test_folded_layer_matches_oracle(name, T, D):
    """moe_layer_forward_fold: the GPU's own routing, folded by the oracle,
    run through the fp64 oracle FFN, matches the GPU layer output; the
    folded batch activates at most D units."""
    wl = WL.ALL[name] if T is None else WL.ALL[name].with_T(T)
    d = make_layer_inputs(wl, DEV)
    desc = B.desc_for(wl, expert_bias=d["expert_bias"])
    S, L = make_fold_tables(wl.E_r, seed=D)
    fold = B.FoldDesc(D=D, S=S.to(DEV), L=L.to(DEV))
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)
    B.check(B.moe_layer_forward_fold(desc, fold, d["x"], d["router_w"], d["w_gate_up"],
                                     d["w_down"], d["k_per_token"], out, st, ws),
            "moe_layer_forward_fold")
    idx = torch.empty(wl.T, wl.k_max, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.k_max, dtype=torch.float32, device=DEV)
    B.check(B.moe_route(desc, d["x"], d["router_w"], None, d["k_per_token"], None, idx, w, st, ws))
    assert B.moe_get_device_status(st) == 0
    fi, fw, fk, pool = F.fold_decode(idx.cpu().numpy(), w.cpu().numpy(),
                                     d["k_per_token"].cpu().numpy(), wl.E_r, D, S.numpy(),
                                     L.numpy())
    assert len(set(fi[fi >= 0].tolist())) <= D
    x = O.bf16_to_f64(bf16_bits(d["x"]))
    wgu, wd = unit_fetch(d["w_gate_up"]), unit_fetch(d["w_down"])
    ref = np.zeros((wl.T, wl.H))
    cache = {}
    for t in range(wl.T):
        for j in range(int(fk[t])):
            u = int(fi[t, j])
            if u not in cache:
                cache[u] = (O.bf16_to_f64(wgu(u)), O.bf16_to_f64(wd(u)))
            ref[t] += float(fw[t, j]) * O.swiglu_ffn(x[t:t + 1], *cache[u])[0]
    assert_close_layer(out.to(torch.float64).cpu().numpy(), ref, f"{wl.name} fold D={D}")
