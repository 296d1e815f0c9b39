"""Thin ctypes binding of libmoe.so, one Python function per C entry point.

Argument marshalling only: tensors are passed as device pointers, streams as
cudaStream_t handles.  Every step of the layer runs in the CUDA library; if
the library is missing or fails to load, every call raises.  The functions
return the moe_status code (an int) and never synchronise, except
``moe_get_device_status``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARGUMENT", 2: "MOE_ERR_UNSUPPORTED_SHAPE",
                3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_TIMEOUT",
                6: "MOE_ERR_NONFINITE", 7: "MOE_ERR_K_RANGE", 8: "MOE_ERR_BAD_INDEX"}
SCORE = {"softmax": 0, "sigmoid": 1}
PATH_AUTO, PATH_PREFILL, PATH_DECODE = 0, 1, 2
DEBUG_SKIP_FIRST_LOAD = 1
DEBUG_FORCE_PAIR = 2

EXPORTS = ("moe_workspace_size", "moe_route", "moe_permute", "moe_gate_up", "moe_down",
           "moe_grouped_ffn", "moe_shared_ffn", "moe_combine", "moe_layer_forward",
           "moe_get_device_status", "moe_status_string", "moe_permute_static",
           "moe_cg_workspace_size", "moe_pack_proxy_rows", "moe_route_cg",
           "moe_layer_forward_cg", "moe_fold_decode", "moe_layer_forward_fold",
           "moe_cost_lookup", "moe_tier_schedule", "moe_layer_forward_paths",
           "moe_layer_forward_host")


class MoeLayerDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("n_sub", ctypes.c_int32), ("I_sub", ctypes.c_int32), ("k_max", ctypes.c_int32),
                ("score", ctypes.c_int), ("renorm", ctypes.c_int32),
                ("route_scale", ctypes.c_float), ("expert_bias", ctypes.c_void_p),
                ("I_shared", ctypes.c_int32), ("w_shared_gate_up", ctypes.c_void_p),
                ("w_shared_down", ctypes.c_void_p), ("path", ctypes.c_int),
                ("debug_flags", ctypes.c_uint32)]


class MoeCgRouter(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int32), ("r", ctypes.c_int32),
                ("router_w_expert", ctypes.c_void_p), ("proxy_w", ctypes.c_void_p),
                ("kappa", ctypes.c_void_p)]


class MoeFoldDesc(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int32), ("pool", ctypes.c_void_p),
                ("unit_scale", ctypes.c_void_p), ("S", ctypes.c_void_p), ("L", ctypes.c_void_p)]


class MoeTierRequest(ctypes.Structure):
    _fields_ = [("arrival", ctypes.c_double), ("n_tokens", ctypes.c_int32), ("k", ctypes.c_int32)]


class MoeCostTable(ctypes.Structure):
    _fields_ = [("n_count", ctypes.c_int32), ("n_points", ctypes.c_void_p),
                ("k_count", ctypes.c_int32), ("k_points", ctypes.c_void_p),
                ("t_us", ctypes.c_void_p)]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")
        self.code = code


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load libmoe.so (raises if it is not built: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libmoe.so is not built ({LIB_PATH}); run "
                               "`python -m aware_moe_expert_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32p = ctypes.c_void_p, ctypes.c_void_p
        D = ctypes.POINTER(MoeLayerDesc)
        sig = {
            "moe_workspace_size": (ctypes.c_size_t, [D]),
            "moe_route": (ctypes.c_int, [D, vp, vp, vp, i32p, vp, i32p, vp, i32p, vp, vp]),
            "moe_permute": (ctypes.c_int, [D, i32p, i32p, i32p, i32p, i32p, i32p, i32p, vp, vp]),
            "moe_permute_static": (ctypes.c_int, [D, i32p, i32p, i32p, i32p, i32p, i32p, i32p,
                                                  vp]),
            "moe_gate_up": (ctypes.c_int, [D, vp, i32p, i32p, vp, vp, i32p, vp, vp]),
            "moe_down": (ctypes.c_int, [D, vp, i32p, vp, vp, i32p, vp, vp]),
            "moe_grouped_ffn": (ctypes.c_int, [D, vp, i32p, i32p, vp, vp, vp, i32p, vp, vp]),
            "moe_shared_ffn": (ctypes.c_int, [D, vp, vp, i32p, vp, vp]),
            "moe_combine": (ctypes.c_int, [D, vp, vp, i32p, vp, i32p, vp, i32p, vp]),
            "moe_layer_forward": (ctypes.c_int, [D, vp, vp, vp, vp, i32p, vp, i32p, vp, vp]),
            "moe_layer_forward_host": (ctypes.c_int, [D, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                      vp, vp, vp]),
            "moe_get_device_status": (ctypes.c_int, [i32p, vp]),
            "moe_cg_workspace_size": (ctypes.c_size_t, [D, ctypes.POINTER(MoeCgRouter)]),
            "moe_pack_proxy_rows": (ctypes.c_int, [D, ctypes.c_int32, vp, i32p, vp, i32p, vp]),
            "moe_route_cg": (ctypes.c_int, [D, ctypes.POINTER(MoeCgRouter), vp, i32p, vp, vp,
                                            i32p, vp, i32p, vp, vp]),
            "moe_layer_forward_cg": (ctypes.c_int, [D, ctypes.POINTER(MoeCgRouter), vp, vp, vp,
                                                    i32p, vp, i32p, vp, vp]),
            "moe_fold_decode": (ctypes.c_int, [D, ctypes.POINTER(MoeFoldDesc), i32p, vp, i32p,
                                               i32p, vp, i32p, i32p, i32p, vp, vp]),
            "moe_layer_forward_fold": (ctypes.c_int, [D, ctypes.POINTER(MoeFoldDesc), vp, vp,
                                                      vp, vp, i32p, vp, i32p, vp, vp]),
            "moe_cost_lookup": (ctypes.c_double, [ctypes.POINTER(MoeCostTable), ctypes.c_double,
                                                  ctypes.c_double]),
            "moe_tier_schedule": (ctypes.c_int32, [ctypes.POINTER(MoeTierRequest), ctypes.c_int32,
                                                   ctypes.c_int32, ctypes.POINTER(MoeCostTable),
                                                   vp, vp, vp, ctypes.c_int32]),
            "moe_layer_forward_paths": (ctypes.c_int, [D, vp, vp, vp, i32p, i32p, vp, i32p, vp,
                                                       i32p, vp, vp]),
            "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


@dataclass
class LayerDesc:
    """Python mirror of moe_layer_desc; tensors kept alive by reference."""
    T: int
    H: int
    n_experts: int
    n_sub: int
    I_sub: int
    k_max: int
    score: str = "softmax"
    renorm: bool = False
    route_scale: float = 1.0
    expert_bias: Optional[torch.Tensor] = None
    I_shared: int = 0
    w_shared_gate_up: Optional[torch.Tensor] = None
    w_shared_down: Optional[torch.Tensor] = None
    debug_flags: int = 0
    path: int = 0              # MOE_PATH_AUTO / PREFILL (1) / DECODE (2)

    @property
    def E_r(self) -> int:
        return self.n_experts * self.n_sub

    def c(self) -> MoeLayerDesc:
        d = MoeLayerDesc()
        d.T, d.H, d.n_experts, d.n_sub = self.T, self.H, self.n_experts, self.n_sub
        d.I_sub, d.k_max = self.I_sub, self.k_max
        d.score = SCORE[self.score]
        d.renorm = int(bool(self.renorm))
        d.route_scale = float(self.route_scale)
        d.expert_bias = _ptr(self.expert_bias)
        d.I_shared = self.I_shared
        d.w_shared_gate_up = _ptr(self.w_shared_gate_up)
        d.w_shared_down = _ptr(self.w_shared_down)
        d.path = int(self.path)
        d.debug_flags = int(self.debug_flags)
        return d


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def desc_for(wl, T=None, expert_bias=None, w_shared_gate_up=None, w_shared_down=None,
             debug_flags=0) -> LayerDesc:
    """LayerDesc for a workload definition (aware_moe_expert_gb300.workloads)."""
    return LayerDesc(T=wl.T if T is None else T, H=wl.H, n_experts=wl.n_experts, n_sub=wl.n_sub,
                     I_sub=wl.I_sub, k_max=wl.k_max, score=wl.score, renorm=wl.renorm,
                     route_scale=wl.route_scale, expert_bias=expert_bias, I_shared=wl.I_shared,
                     w_shared_gate_up=w_shared_gate_up, w_shared_down=w_shared_down,
                     debug_flags=debug_flags)


def moe_workspace_size(desc: LayerDesc) -> int:
    d = desc.c()
    return int(lib().moe_workspace_size(ctypes.byref(d)))


def moe_route(desc, x, router_w, logits_in, k_per_token, logits_out, topk_idx, topk_w,
              dev_status, workspace, stream=None) -> int:
    d = desc.c()
    return lib().moe_route(ctypes.byref(d), _ptr(x), _ptr(router_w), _ptr(logits_in),
                           _ptr(k_per_token), _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w),
                           _ptr(dev_status), _ptr(workspace), _stream(stream))


def moe_permute(desc, topk_idx, k_per_token, counts, offsets, sorted_token, inv_row, dev_status,
                workspace, stream=None) -> int:
    d = desc.c()
    return lib().moe_permute(ctypes.byref(d), _ptr(topk_idx), _ptr(k_per_token), _ptr(counts),
                             _ptr(offsets), _ptr(sorted_token), _ptr(inv_row), _ptr(dev_status),
                             _ptr(workspace), _stream(stream))


def moe_permute_static(desc, topk_idx, k_per_token, counts, offsets, sorted_token, inv_row,
                       dev_status, stream=None) -> int:
    """moe_permute with its scratch in the library's own device array (no
    workspace argument, nothing allocated)."""
    d = desc.c()
    return lib().moe_permute_static(ctypes.byref(d), _ptr(topk_idx), _ptr(k_per_token),
                                    _ptr(counts), _ptr(offsets), _ptr(sorted_token),
                                    _ptr(inv_row), _ptr(dev_status), _stream(stream))


def moe_gate_up(desc, x, sorted_token, offsets, w_gate_up, act, dev_status, workspace,
                stream=None) -> int:
    d = desc.c()
    return lib().moe_gate_up(ctypes.byref(d), _ptr(x), _ptr(sorted_token), _ptr(offsets),
                             _ptr(w_gate_up), _ptr(act), _ptr(dev_status), _ptr(workspace),
                             _stream(stream))


def moe_down(desc, act, offsets, w_down, y_perm, dev_status, workspace, stream=None) -> int:
    d = desc.c()
    return lib().moe_down(ctypes.byref(d), _ptr(act), _ptr(offsets), _ptr(w_down), _ptr(y_perm),
                          _ptr(dev_status), _ptr(workspace), _stream(stream))


def moe_grouped_ffn(desc, x, sorted_token, offsets, w_gate_up, w_down, y_perm, dev_status,
                    workspace, stream=None) -> int:
    d = desc.c()
    return lib().moe_grouped_ffn(ctypes.byref(d), _ptr(x), _ptr(sorted_token), _ptr(offsets),
                                 _ptr(w_gate_up), _ptr(w_down), _ptr(y_perm), _ptr(dev_status),
                                 _ptr(workspace), _stream(stream))


def moe_shared_ffn(desc, x, y_shared, dev_status, workspace, stream=None) -> int:
    d = desc.c()
    return lib().moe_shared_ffn(ctypes.byref(d), _ptr(x), _ptr(y_shared), _ptr(dev_status),
                                _ptr(workspace), _stream(stream))


def moe_combine(desc, y_perm, y_shared, inv_row, topk_w, k_per_token, out, dev_status,
                stream=None) -> int:
    d = desc.c()
    return lib().moe_combine(ctypes.byref(d), _ptr(y_perm), _ptr(y_shared), _ptr(inv_row),
                             _ptr(topk_w), _ptr(k_per_token), _ptr(out), _ptr(dev_status),
                             _stream(stream))


def moe_layer_forward(desc, x, router_w, w_gate_up, w_down, k_per_token, out, dev_status,
                      workspace, stream=None) -> int:
    """desc: a LayerDesc, or the MoeLayerDesc its c() returned (a serving loop
    can build that once and skip the conversion on every call)."""
    d = desc if isinstance(desc, MoeLayerDesc) else desc.c()
    return lib().moe_layer_forward(ctypes.byref(d), _ptr(x), _ptr(router_w), _ptr(w_gate_up),
                                   _ptr(w_down), _ptr(k_per_token), _ptr(out), _ptr(dev_status),
                                   _ptr(workspace), _stream(stream))


def moe_layer_forward_host(desc, x_host, k_host, out_host, x_dev, k_dev, out_dev, router_w,
                           w_gate_up, w_down, dev_status, workspace, stream=None) -> int:
    """x_host, k_host, out_host: CPU tensors (pinned for an asynchronous call)
    or raw host addresses; the rest as for moe_layer_forward."""
    d = desc if isinstance(desc, MoeLayerDesc) else desc.c()
    return lib().moe_layer_forward_host(ctypes.byref(d), _ptr(x_host), _ptr(k_host),
                                        _ptr(out_host), _ptr(x_dev), _ptr(k_dev), _ptr(out_dev),
                                        _ptr(router_w), _ptr(w_gate_up), _ptr(w_down),
                                        _ptr(dev_status), _ptr(workspace), _stream(stream))


@dataclass
class CgRouter:
    """Python mirror of moe_cg_router (the training-free proxy router)."""
    m: int
    r: int
    router_w_expert: torch.Tensor      # bf16 [n_experts, H]
    proxy_w: torch.Tensor              # bf16 [E_r * 2 * r, H] (moe_pack_proxy_rows)
    kappa: torch.Tensor                # int32 [k_max + 1, m] on the device

    def c(self) -> MoeCgRouter:
        g = MoeCgRouter()
        g.m, g.r = int(self.m), int(self.r)
        g.router_w_expert = _ptr(self.router_w_expert)
        g.proxy_w = _ptr(self.proxy_w)
        g.kappa = _ptr(self.kappa)
        return g


def moe_cg_workspace_size(desc: LayerDesc, cg: CgRouter) -> int:
    d, g = desc.c(), cg.c()
    return int(lib().moe_cg_workspace_size(ctypes.byref(d), ctypes.byref(g)))


def moe_pack_proxy_rows(desc, r, w_gate_up, gate_neurons, proxy_w, dev_status,
                        stream=None) -> int:
    d = desc.c()
    return lib().moe_pack_proxy_rows(ctypes.byref(d), int(r), _ptr(w_gate_up),
                                     _ptr(gate_neurons), _ptr(proxy_w), _ptr(dev_status),
                                     _stream(stream))


def moe_route_cg(desc, cg, x, k_per_token, expert_logits_out, proxy_out, topk_idx, topk_w,
                 dev_status, workspace, stream=None) -> int:
    d, g = desc.c(), cg.c()
    return lib().moe_route_cg(ctypes.byref(d), ctypes.byref(g), _ptr(x), _ptr(k_per_token),
                              _ptr(expert_logits_out), _ptr(proxy_out), _ptr(topk_idx),
                              _ptr(topk_w), _ptr(dev_status), _ptr(workspace), _stream(stream))


def moe_layer_forward_cg(desc, cg, x, w_gate_up, w_down, k_per_token, out, dev_status,
                         workspace, stream=None) -> int:
    d, g = desc.c(), cg.c()
    return lib().moe_layer_forward_cg(ctypes.byref(d), ctypes.byref(g), _ptr(x),
                                      _ptr(w_gate_up), _ptr(w_down), _ptr(k_per_token),
                                      _ptr(out), _ptr(dev_status), _ptr(workspace),
                                      _stream(stream))


@dataclass
class FoldDesc:
    """Python mirror of moe_fold_desc (decode expert-pool folding)."""
    D: int
    S: torch.Tensor                          # fp32 [E_r, E_r]
    L: torch.Tensor                          # fp32 [E_r, E_r]
    pool: Optional[torch.Tensor] = None      # int32 [D]: static pool; None: dynamic
    unit_scale: Optional[torch.Tensor] = None

    def c(self) -> MoeFoldDesc:
        f = MoeFoldDesc()
        f.D = int(self.D)
        f.pool = _ptr(self.pool)
        f.unit_scale = _ptr(self.unit_scale)
        f.S = _ptr(self.S)
        f.L = _ptr(self.L)
        return f


def moe_fold_decode(desc, fold, topk_idx, topk_w, k_per_token, topk_idx_out, topk_w_out, k_out,
                    pool_out, dev_status, workspace, stream=None) -> int:
    d, f = desc.c(), fold.c()
    return lib().moe_fold_decode(ctypes.byref(d), ctypes.byref(f), _ptr(topk_idx), _ptr(topk_w),
                                 _ptr(k_per_token), _ptr(topk_idx_out), _ptr(topk_w_out),
                                 _ptr(k_out), _ptr(pool_out), _ptr(dev_status), _ptr(workspace),
                                 _stream(stream))


def moe_layer_forward_fold(desc, fold, x, router_w, w_gate_up, w_down, k_per_token, out,
                           dev_status, workspace, stream=None) -> int:
    d, f = desc.c(), fold.c()
    return lib().moe_layer_forward_fold(ctypes.byref(d), ctypes.byref(f), _ptr(x), _ptr(router_w),
                                        _ptr(w_gate_up), _ptr(w_down), _ptr(k_per_token),
                                        _ptr(out), _ptr(dev_status), _ptr(workspace),
                                        _stream(stream))


class CostTable:
    """Host mirror of moe_cost_table: T(n, k) in microseconds at token buckets
    n_points and budget buckets k_points (t_us[k_index][n_index])."""

    def __init__(self, n_points, k_points, t_us):
        import numpy as np
        self.n = np.ascontiguousarray(n_points, dtype=np.int32)
        self.k = np.ascontiguousarray(k_points, dtype=np.int32)
        self.t = np.ascontiguousarray(t_us, dtype=np.float64).reshape(len(self.k), len(self.n))

    def c(self) -> MoeCostTable:
        c = MoeCostTable()
        c.n_count, c.k_count = len(self.n), len(self.k)
        c.n_points = self.n.ctypes.data
        c.k_points = self.k.ctypes.data
        c.t_us = self.t.ctypes.data
        return c


def moe_cost_lookup(table: CostTable, n: float, k: float) -> float:
    c = table.c()
    return float(lib().moe_cost_lookup(ctypes.byref(c), float(n), float(k)))


def moe_tier_schedule(requests, M: int, table: CostTable):
    """requests: sequence of (arrival, n_tokens, k).  Returns (batch_of,
    batch_k, batch_tokens) as lists, or raises on an error code."""
    import numpy as np
    n = len(requests)
    arr = (MoeTierRequest * max(n, 1))()
    for i, (a, tok, k) in enumerate(requests):
        arr[i].arrival, arr[i].n_tokens, arr[i].k = float(a), int(tok), int(k)
    batch_of = np.zeros(max(n, 1), dtype=np.int32)
    bk = np.zeros(max(n, 1), dtype=np.int32)
    bt = np.zeros(max(n, 1), dtype=np.int32)
    c = table.c()
    nb = lib().moe_tier_schedule(arr, n, int(M), ctypes.byref(c), batch_of.ctypes.data,
                                 bk.ctypes.data, bt.ctypes.data, max(n, 1))
    if nb < 0:
        raise MoeError(1, f"moe_tier_schedule returned {nb}")
    return batch_of[:n].tolist(), bk[:nb].tolist(), bt[:nb].tolist()


def moe_layer_forward_paths(desc, x, w_gate_up, w_down, src_idx, tgt_idx, beta, n_paths, out,
                            dev_status, workspace, stream=None) -> int:
    d = desc.c()
    return lib().moe_layer_forward_paths(ctypes.byref(d), _ptr(x), _ptr(w_gate_up), _ptr(w_down),
                                         _ptr(src_idx), _ptr(tgt_idx), _ptr(beta),
                                         _ptr(n_paths), _ptr(out), _ptr(dev_status),
                                         _ptr(workspace), _stream(stream))


def moe_get_device_status(dev_status, stream=None) -> int:
    return lib().moe_get_device_status(_ptr(dev_status), _stream(stream))


def moe_status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def check(code: int, where: str = "moe") -> None:
    if code != MOE_OK:
        raise MoeError(code, where)


class MoeLayer:
    """Convenience owner of the workspace and status word for one layer shape
    on one device; every call goes straight to the C ABI."""

    def __init__(self, desc: LayerDesc, device="cuda"):
        self.desc = desc
        self.device = torch.device(device)
        n = moe_workspace_size(desc)
        if n == 0:
            raise MoeError(2, "moe_workspace_size")
        self.workspace = torch.empty(n, dtype=torch.uint8, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    def forward(self, x, router_w, w_gate_up, w_down, k_per_token, out=None, stream=None):
        if out is None:
            out = torch.empty(self.desc.T, self.desc.H, dtype=torch.bfloat16, device=self.device)
        check(moe_layer_forward(self.desc, x, router_w, w_gate_up, w_down, k_per_token, out,
                                self.status, self.workspace, stream), "moe_layer_forward")
        return out

    def device_status(self, stream=None) -> int:
        return moe_get_device_status(self.status, stream)
