"""The weighted combine (MoE-Prism §III-B2: a token's output is the
gate-weighted sum of its selected units' FFN outputs) through moe_combine.

Batches of 32 tokens and more, up to one resident wave, run the kernel that
loads a token's indices and rows in two round trips; smaller batches run the
one that loads them four at a time.  Both add the rows in j order with fmaf
from 0 and round once, so on the same tokens they agree bit for bit; a 64-token
call is compared with four 16-token calls on the same rows.  Rows outside
y_perm are reported and skipped."""
import numpy as np
import pytest
import torch

from aware_moe_expert_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(T, H, k_max, seed, n_slices):
    """Per slice of T / n_slices tokens: its own block of y_perm rows, so a
    slice can also be combined on its own."""
    rng = np.random.default_rng(seed)
    Ts = T // n_slices
    rows_per = Ts * k_max
    y = torch.from_numpy(rng.standard_normal((T * k_max, H)).astype(np.float32)).to(torch.bfloat16)
    k = rng.integers(1, k_max + 1, size=T).astype(np.int32)
    inv = np.full((T, k_max), -1, dtype=np.int32)
    w = np.zeros((T, k_max), dtype=np.float32)
    for s in range(n_slices):
        perm = rng.permutation(rows_per)
        pos = 0
        for t in range(s * Ts, (s + 1) * Ts):
            inv[t, :k[t]] = perm[pos:pos + k[t]]       # rows local to the slice
            pos += k[t]
            w[t, :k[t]] = rng.random(k[t]).astype(np.float32)
    return y.to(DEV), torch.from_numpy(inv).to(DEV), torch.from_numpy(w).to(DEV), \
        torch.from_numpy(k).to(DEV)


@pytest.mark.parametrize("k_max", [8, 16])
def test_wide_combine_equals_the_four_at_a_time_combine(k_max):
    T, H, n = 64, 2048, 4
    Ts = T // n
    y, inv, w, k = _case(T, H, k_max, 7 + k_max, n)
    # whole batch: slice s's rows sit at s * Ts * k_max in y_perm
    inv_all = inv.clone()
    for s in range(n):
        blk = inv_all[s * Ts:(s + 1) * Ts]
        blk[blk >= 0] += s * Ts * k_max
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    B.check(B.moe_combine(B.LayerDesc(T=T, H=H, n_experts=64, n_sub=1, I_sub=64, k_max=k_max),
                          y, None, inv_all, w, k, out, st), "moe_combine")
    assert B.moe_get_device_status(st) == 0
    ref = torch.empty_like(out)
    d16 = B.LayerDesc(T=Ts, H=H, n_experts=64, n_sub=1, I_sub=64, k_max=k_max)
    for s in range(n):
        B.check(B.moe_combine(d16, y[s * Ts * k_max:(s + 1) * Ts * k_max], None,
                              inv[s * Ts:(s + 1) * Ts].contiguous(),
                              w[s * Ts:(s + 1) * Ts].contiguous(), k[s * Ts:(s + 1) * Ts].contiguous(),
                              ref[s * Ts:(s + 1) * Ts], st), "moe_combine")
    assert B.moe_get_device_status(st) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # and against the definition in float64
    yd = y.double().cpu().numpy()
    want = np.zeros((T, H))
    iv, wv, kv = inv_all.cpu().numpy(), w.cpu().numpy(), k.cpu().numpy()
    for t in range(T):
        for j in range(kv[t]):
            want[t] += float(wv[t, j]) * yd[iv[t, j]]
    got = out.double().cpu().numpy()
    assert np.all(np.abs(got - want) <= 1e-2 + 1e-2 * np.abs(want))


@pytest.mark.parametrize("T", [16, 64])
def test_combine_reports_rows_outside_y_perm(T):
    H, k_max = 256, 8
    y, inv, w, k = _case(T, H, k_max, 3, 1)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    desc = B.LayerDesc(T=T, H=H, n_experts=64, n_sub=1, I_sub=64, k_max=k_max)
    ref = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    bad = inv.clone()
    t_bad = int(np.nonzero(k.cpu().numpy() >= 2)[0][-1])   # a token with two rows at least
    bad[t_bad, 0] = T * k_max                 # one past the last row
    inv_ok = bad.clone()
    w_ok = w.clone()
    w_ok[t_bad, 0] = 0.0                      # the skipped row adds nothing
    inv_ok[t_bad, 0] = inv_ok[t_bad, 1]
    B.check(B.moe_combine(desc, y, None, inv_ok, w_ok, k, ref, st), "moe_combine")
    assert B.moe_get_device_status(st) == 0
    out = torch.empty_like(ref)
    B.check(B.moe_combine(desc, y, None, bad, w, k, out, st), "moe_combine")
    assert B.moe_get_device_status(st) == 8    # MOE_ERR_BAD_INDEX
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
