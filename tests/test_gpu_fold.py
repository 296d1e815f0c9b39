"""GPU parity of decode expert-pool folding (moe_fold_decode,
moe_layer_forward_fold) against the CPU oracle (oracle/exfold.py).

The oracle scores units by their exact (float64) aggregate routed weight; the
GPU adds the same fp32 weights in fp32.  The pool must equal the oracle's,
except where a differing unit's exact score lies within the fp32 summation
bound of the selection boundary (a near tie, either choice correct).  Given
the GPU's pool, targets and new budgets must equal the oracle's exactly and
merged weights agree within the fp32 bound of their terms.  The folded
layer's output is compared, in the stated layer tolerance, with the fp64
oracle FFN over the folded routing of the GPU's own route.
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
    n_np, w_np, k_np = idx.numpy(), w.numpy(), k.numpy()
    if pool_in is None:
        want_pool = F.select_pool(F.pool_scores(n_np, w_np, k_np, E_r), D)
        gpu_pool = pool[:len(want_pool)]
        n_tied = _check_pool_near_ties(n_np, w_np, k_np, E_r, D, gpu_pool, want_pool)
        assert n_tied <= 2, f"{n_tied} pool members differ"
    else:
        gpu_pool = pool[:D]
        np.testing.assert_array_equal(np.sort(gpu_pool), np.sort(pool_in.numpy()))
    wi, ww, wk, _, (mag, nt) = F.fold_decode(n_np, w_np, k_np, E_r, D, S.numpy(), L.numpy(),
                                             pool=gpu_pool, return_abs=True)
    np.testing.assert_array_equal(ok, wk)
    np.testing.assert_array_equal(oi, wi)
    # an fp32 product per route and fp32 additions of the merged terms
    bound = np.vectorize(F.gamma)(nt + 1) * mag
    assert (np.abs(ow.astype(np.float64) - ww) <= bound).all()


def _check_pool_near_ties(idx, w, k, E_r, D, gpu_pool, want_pool):
    """A unit in one pool but not the other must lie within the summation
    bounds of the boundary between the D-th and (D+1)-th exact scores."""
    got, want = set(int(u) for u in gpu_pool), set(int(u) for u in want_pool)
    if got == want:
        return 0
    sc = F.pool_scores(idx, w, k, E_r)
    bd = F.score_error_bound(idx, w, k, E_r)
    order = sorted(range(E_r), key=lambda u: (-sc[u], u))
    hi = sc[order[D - 1]]                      # the D-th exact score
    lo = sc[order[D]] if D < E_r else hi       # the (D+1)-th
    for u in got ^ want:
        # u can trade places with a unit across the boundary only if their
        # fp32 evaluations can cross: within u's bound plus the largest other
        margin = bd[u] + bd.max()
        assert hi - margin <= sc[u] <= lo + margin, (u, sc[u], lo, hi, margin)
    return len(got ^ want) // 2


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
    # the GPU's pool for this routing (the layer's own fold kernels), checked
    # against the exact-score pool up to near ties, then used by the oracle
    i_np, w_np, k_np = idx.cpu().numpy(), w.cpu().numpy(), d["k_per_token"].cpu().numpy()
    *_, gpu_pool, code = _run_fold(desc, fold, idx.cpu(), w.cpu(), d["k_per_token"].cpu())
    assert code == 0
    want_pool = F.select_pool(F.pool_scores(i_np, w_np, k_np, wl.E_r), D)
    assert _check_pool_near_ties(i_np, w_np, k_np, wl.E_r, D, gpu_pool[:D], want_pool) <= 2
    fi, fw, fk, pool = F.fold_decode(i_np, w_np, k_np, wl.E_r, D, S.numpy(), L.numpy(),
                                     pool=gpu_pool[:D])
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
