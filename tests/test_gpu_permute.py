"""GPU parity of the permutation: counts, offsets, sorted_token and inv_row
bit-exact against the oracle, on routings with ragged, empty and full units."""
import numpy as np
import pytest
import torch

from aware_moe_expert_gb300 import binding as B
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _random_routing(T, E_r, k_max, seed, skew=0.0):
    rng = np.random.default_rng(seed)
    k = rng.integers(1, k_max + 1, size=T).astype(np.int32)
    idx = np.full((T, k_max), -1, dtype=np.int32)
    p = np.exp(-skew * np.log(np.arange(1, E_r + 1)))
    p /= p.sum()
    for t in range(T):
        idx[t, :k[t]] = rng.choice(E_r, size=k[t], replace=False, p=p)
    return idx, k


def _gpu_permute(desc, idx, k):
    T, E_r, k_max = desc.T, desc.E_r, desc.k_max
    d_idx = torch.from_numpy(idx).to(DEV)
    d_k = torch.from_numpy(k).to(DEV)
    counts = torch.full((E_r,), -5, dtype=torch.int32, device=DEV)
    offsets = torch.full((E_r + 1,), -5, dtype=torch.int32, device=DEV)
    st_tok = torch.full((max(T * k_max, 1),), -5, dtype=torch.int32, device=DEV)
    inv = torch.full((max(T * k_max, 1),), -5, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    B.check(B.moe_permute(desc, d_idx, d_k, counts, offsets, st_tok, inv, st, ws), "moe_permute")
    code = B.moe_get_device_status(st)
    return (counts.cpu().numpy(), offsets.cpu().numpy(), st_tok.cpu().numpy(),
            inv.cpu().numpy()[: T * k_max].reshape(T, k_max), code)


@pytest.mark.parametrize("T,E_r,k_max,skew", [(1, 8, 4, 0.0), (31, 64, 8, 0.0), (32, 64, 8, 0.0),
                                              (33, 64, 8, 0.0), (1000, 128, 8, 1.1),
                                              (1024, 256, 16, 0.0), (4097, 32, 8, 2.0),
                                              (16384, 256, 8, 0.5), (70, 3, 3, 0.0),
                                              # scatter CTAs of 256 slots spanning one
                                              # bitmap word (k_max 8), half a word (16),
                                              # several words (k_max 1, 2, 3)
                                              (8192, 128, 8, 1.1), (2048, 256, 1, 0.0),
                                              (3072, 64, 2, 0.7), (4096, 256, 8, 0.0),
                                              (2048, 48, 3, 0.0), (1024, 33, 5, 0.0),
                                              # the one-CTA kernel's last size and the
                                              # bitmap kernels' first ones
                                              (128, 256, 16, 0.0), (129, 256, 16, 0.0),
                                              (200, 128, 8, 1.1), (256, 256, 32, 0.0)])
def test_permute_bit_exact(T, E_r, k_max, skew):
    idx, k = _random_routing(T, E_r, k_max, seed=T + E_r, skew=skew)
    desc = B.LayerDesc(T=T, H=64, n_experts=E_r, n_sub=1, I_sub=64, k_max=k_max)
    counts, offsets, st_tok, inv, code = _gpu_permute(desc, idx, k)
    assert code == 0, B.STATUS_NAMES[code]
    wc, wo, wst, winv = O.permute(idx, k, E_r)
    np.testing.assert_array_equal(counts, wc)
    np.testing.assert_array_equal(offsets, wo)
    n = int(wo[-1])
    np.testing.assert_array_equal(st_tok[:n], wst)
    np.testing.assert_array_equal(inv, winv)


def test_permute_empty_batch_gives_zero_offsets():
    desc = B.LayerDesc(T=0, H=64, n_experts=16, n_sub=1, I_sub=64, k_max=4)
    offsets = torch.full((17,), -5, dtype=torch.int32, device=DEV)
    counts = torch.full((16,), -5, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(B.moe_workspace_size(desc), 256), dtype=torch.uint8, device=DEV)
    dummy = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.check(B.moe_permute(desc, dummy, dummy, counts, offsets, dummy, dummy, st, ws))
    assert B.moe_get_device_status(st) == 0
    assert (offsets.cpu().numpy() == 0).all() and (counts.cpu().numpy() == 0).all()


def test_permute_reports_bad_unit_index():
    T, E_r, k_max = 40, 16, 3
    idx, k = _random_routing(T, E_r, k_max, seed=1)
    idx[5, 0] = E_r          # out of range
    desc = B.LayerDesc(T=T, H=64, n_experts=E_r, n_sub=1, I_sub=64, k_max=k_max)
    *_, code = _gpu_permute(desc, idx, k)
    assert code == 8  # MOE_ERR_BAD_INDEX
    idx, k = _random_routing(T, E_r, k_max, seed=2)
    k[7] = 3
    idx[7, :3] = [4, 9, 4]   # repeated unit within a token
    *_, code = _gpu_permute(desc, idx, k)
    assert code == 8
