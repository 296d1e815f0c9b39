"""The C ABI without a GPU: the library builds, loads, exports every function
include/moe.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

from aware_moe_expert_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from aware_moe_expert_gb300 import build
        build.build()
    return B.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(moe_[a-z_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_binding_exports():
    assert sorted(declared_functions()) == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code, name in B.STATUS_NAMES.items():
        assert B.moe_status_string(code) == name
    assert B.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def _desc(**kw):
    base = dict(T=64, H=256, n_experts=16, n_sub=4, I_sub=128, k_max=8)
    base.update(kw)
    return B.LayerDesc(**base)


@pytest.mark.parametrize("kw,expect_zero", [
    (dict(), False),
    (dict(H=100), True),                 # H % 64
    (dict(I_sub=96), True),              # I_sub % 64
    (dict(n_experts=65, n_sub=4), True),  # E_r > 256
    (dict(k_max=33, n_experts=64), True),  # k_max > 32
    (dict(k_max=0), True),
    (dict(T=-1), True),
    (dict(T=0), False),
])
def test_workspace_size_validates_shapes(lib, kw, expect_zero):
    n = B.moe_workspace_size(_desc(**kw))
    assert (n == 0) == expect_zero
    if not expect_zero:
        assert n % 256 == 0


def test_workspace_grows_with_tokens(lib):
    assert B.moe_workspace_size(_desc(T=128)) > B.moe_workspace_size(_desc(T=64))


def test_host_rejects_bad_arguments_without_a_gpu(lib):
    d = _desc()
    fake = 1 << 20          # aligned but never dereferenced: validation fails first
    ws = 1 << 21
    # unsupported shape
    assert B.moe_layer_forward(_desc(H=100), fake, fake, fake, fake, fake, fake, fake, ws, 0) == 2
    # null pointers
    assert B.moe_layer_forward(d, None, fake, fake, fake, fake, fake, fake, ws, 0) == 1
    assert B.moe_route(d, None, None, None, fake, None, fake, fake, fake, ws, 0) == 1
    assert B.moe_combine(d, fake, None, None, fake, fake, fake, fake, 0) == 1
    # misaligned bf16 pointer
    assert B.moe_grouped_ffn(d, fake + 2, fake, fake, fake, fake, fake, fake, ws, 0) == 1
    # workspace missing or misaligned
    assert B.moe_layer_forward(d, fake, fake, fake, fake, fake, fake, fake, None, 0) == 3


def test_host_buffer_forward_rejects_bad_arguments_before_copying(lib):
    """moe_layer_forward_host checks the descriptor, the host and device
    pointers and the workspace on the host, before any copy is enqueued."""
    d = _desc()
    fake = 1 << 20                      # aligned, never dereferenced
    ws = 1 << 21
    args = [fake] * 9                   # x_host, k_host, out_host, x_dev, k_dev, out_dev, weights
    assert B.moe_layer_forward_host(_desc(H=100), *args, fake, ws, 0) == 2
    assert B.moe_layer_forward_host(d, None, *args[1:], fake, ws, 0) == 1
    assert B.moe_layer_forward_host(d, *args[:3], None, *args[4:], fake, ws, 0) == 1
    assert B.moe_layer_forward_host(d, *args, None, ws, 0) == 1
    assert B.moe_layer_forward_host(d, *args, fake, None, 0) == 3
    assert B.moe_layer_forward_host(_desc(T=0), *args, fake, ws, 0) == 0
    assert B.moe_layer_forward(d, fake, fake, fake, fake, fake, fake, fake, ws + 16, 0) == 3
    # shared expert requested without weights
    assert B.moe_shared_ffn(_desc(), fake, fake, fake, ws, 0) == 1
    assert B.moe_workspace_size(_desc(I_shared=128)) == 0
    assert B.moe_get_device_status(None, 0) == 1


def _cg(m=2, r=4):
    fake = 1 << 20
    return B.CgRouter(m=m, r=r, router_w_expert=fake, proxy_w=fake, kappa=fake)


@pytest.mark.parametrize("kw,cg_kw,expect_zero", [
    (dict(), dict(), False),
    (dict(), dict(m=0), True),                       # m < 1
    (dict(), dict(m=17), True),                      # m > n_experts
    (dict(), dict(r=0), True),
    (dict(), dict(r=129), True),                     # r > I_sub
    (dict(n_experts=2, n_sub=33, k_max=8), dict(), True),   # n_sub > 32
    (dict(k_max=9), dict(m=2), True),                # k_max > m * n_sub
])
def test_cg_workspace_size_validates(lib, kw, cg_kw, expect_zero):
    n = B.moe_cg_workspace_size(_desc(**kw), _cg(**cg_kw))
    assert (n == 0) == expect_zero
    if not expect_zero:
        assert n > B.moe_workspace_size(_desc(**kw)) and n % 256 == 0


def test_cg_calls_reject_bad_arguments_without_a_gpu(lib):
    d, fake, ws = _desc(), 1 << 20, 1 << 21
    assert B.moe_route_cg(d, _cg(m=0), fake, fake, None, None, fake, fake, fake, ws, 0) == 2
    assert B.moe_route_cg(d, _cg(), None, fake, None, None, fake, fake, fake, ws, 0) == 1
    assert B.moe_route_cg(d, _cg(), fake, fake, None, None, fake, fake, fake, None, 0) == 3
    assert B.moe_pack_proxy_rows(d, 0, fake, fake, fake, fake, 0) == 2
    assert B.moe_pack_proxy_rows(d, 4, fake + 2, fake, fake, fake, 0) == 1
    assert B.moe_layer_forward_cg(d, _cg(), fake, fake, fake, fake, fake, fake, ws + 16, 0) == 3


def test_cg_rejects_too_many_proxy_pairs(lib):
    # m * n_sub * r = 4 * 4 * 129 > 2048
    assert B.moe_cg_workspace_size(_desc(I_sub=256), _cg(m=4, r=129)) == 0
    assert B.moe_cg_workspace_size(_desc(I_sub=256), _cg(m=4, r=128)) > 0


@pytest.mark.parametrize("kw,status", [(dict(T=-1), 1), (dict(k_max=0), 1), (dict(H=100), 2),
                                       (dict(n_experts=65, n_sub=4), 2)])
def test_static_scratch_permute_reports_what_moe_permute_reports(lib, kw, status):
    """moe_permute_static checks the descriptor exactly as moe_permute does,
    before any CUDA call: invalid (1) and unsupported (2) descriptors give
    the same status from both."""
    fake = 1 << 20
    ws = 1 << 21
    d = _desc(**kw)
    assert B.moe_permute(d, fake, fake, fake, fake, fake, fake, fake, ws, 0) == status
    assert B.moe_permute_static(d, fake, fake, fake, fake, fake, fake, fake, 0) == status
