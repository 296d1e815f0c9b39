"""moe_permute_static: the permutation for callers that cannot allocate.

Some callers cannot hand the library a workspace: they route tokens inside a
serving loop that must stay out of the allocator, or from a plug-in that owns
no device buffers.
moe_permute_static keeps its scratch in the library's own device array; this
checks, through the C ABI, that it returns exactly what moe_permute (with a
workspace) returns, on two different routings in a row (so nothing left in
the shared array from the first call leaks into the second), and that a
batch too large for the array is refused.  Collected last on purpose.
"""
import numpy as np
import pytest
import torch

from aware_moe_expert_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _routing(T, E_r, k_max, seed):
    rng = np.random.default_rng(seed)
    k = rng.integers(1, k_max + 1, size=T).astype(np.int32)
    idx = np.full((T, k_max), -1, dtype=np.int32)
    for t in range(T):
        idx[t, :k[t]] = rng.choice(E_r, size=k[t], replace=False)
    return torch.from_numpy(idx).to(DEV), torch.from_numpy(k).to(DEV)


def _outputs(T, E_r, k_max):
    return (torch.full((E_r,), -9, dtype=torch.int32, device=DEV),
            torch.full((E_r + 1,), -9, dtype=torch.int32, device=DEV),
            torch.full((T * k_max,), -9, dtype=torch.int32, device=DEV),
            torch.full((T * k_max,), -9, dtype=torch.int32, device=DEV),
            torch.zeros(1, dtype=torch.int32, device=DEV))


# (16384, 256, 8) is the exact-fit boundary: 2 * 256 units * 512 words * 4 bytes
# = 1 MiB, the whole array (one token more is refused, below).
@pytest.mark.parametrize("T,E_r,k_max", [(300, 256, 8),
                                         pytest.param(16384, 256, 8, id="exact-fit-1MiB"),
                                         (4097, 32, 8), (100, 64, 8)])
def test_static_scratch_permute_matches_workspace_permute(T, E_r, k_max):
    desc = B.LayerDesc(T=T, H=64, n_experts=E_r, n_sub=1, I_sub=64, k_max=k_max)
    ws = torch.empty(B.moe_workspace_size(desc), dtype=torch.uint8, device=DEV)
    for call, seed in enumerate((T + 1, T + 2)):      # two calls in a row, different routings
        idx, k = _routing(T, E_r, k_max, seed)
        ref = _outputs(T, E_r, k_max)
        got = _outputs(T, E_r, k_max)
        B.check(B.moe_permute(desc, idx, k, *ref[:4], ref[4], ws), "moe_permute")
        B.check(B.moe_permute_static(desc, idx, k, *got[:4], got[4]), "moe_permute_static")
        assert B.moe_get_device_status(ref[4]) == 0
        assert B.moe_get_device_status(got[4]) == 0
        n = int(ref[1][-1].item())
        assert n == int(k.sum().item())
        for name, a, b in zip(("counts", "offsets", "sorted_token", "inv_row"), ref[:4], got[:4]):
            if name == "sorted_token":
                a, b = a[:n], b[:n]
            assert torch.equal(a, b), f"call {call}: {name} differs"


def test_static_scratch_permute_refuses_batches_beyond_its_array():
    # 2 * 256 units * ceil(16385 / 32) words * 4 bytes > 1 MiB
    desc = B.LayerDesc(T=16385, H=64, n_experts=256, n_sub=1, I_sub=64, k_max=8)
    idx, k = _routing(8, 256, 8, 0)          # never read: refused on the host
    out = _outputs(8, 256, 8)
    assert B.moe_permute_static(desc, idx, k, *out[:4], out[4]) == 2  # MOE_ERR_UNSUPPORTED_SHAPE
