"""Python binding of the ds4moe C ABI (``include/ds4moe.h``).

Argument marshalling only: every step of the layer runs in the CUDA library
``libds4moe.so`` built from ``csrc/`` for sm_103a. Importing this package
fails loudly when that library is missing; there is no fallback.

The raw entry points keep the C names (``ds4moe_create``, ``ds4moe_route``,
``ds4moe_forward`` ...) and take torch tensors or raw device addresses.
``MoELayer`` wraps a handle for callers holding torch tensors.
"""
from __future__ import annotations

import ctypes
import os

from ._build import INCLUDE, LIB_PATH, NVCC_FLAGS, build, sources  # noqa: F401

DS4MOE_MAGIC = 0x454D3444
DS4MOE_VERSION = 3
DS4MOE_OK, DS4MOE_EINVAL, DS4MOE_ENOMEM, DS4MOE_ECUDA, DS4MOE_EUNSUPPORTED, DS4MOE_ETIMEOUT, DS4MOE_EDEVICE = (
    0, -1, -2, -3, -4, -5, -6)
DS4MOE_ESCRATCH = -7
DS4MOE_NOALLOC_SCRATCH = 4 << 20
PATH_AUTO, PATH_DECODE, PATH_PREFILL, PATH_BATCH = 0, 1, 2, 3
AUTO_DECODE_MAX_T = 1
AUTO_BATCH_MAX_T = 64
AUTO_MX4_PREFILL_MIN_T = 3
AUTO_VQ_PREFILL_MIN_T = 1
BATCH_MAX_T = 64
FLAG_MXFP4 = 1
FLAG_VQ12, FLAG_VQ13 = 2, 4


class LayerDesc(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_uint32), ("version", ctypes.c_uint32), ("hidden", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class Weights(ctypes.Structure):
    _fields_ = [("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p), ("gate", ctypes.c_void_p),
                ("up", ctypes.c_void_p), ("down", ctypes.c_void_p), ("sh_gate", ctypes.c_void_p),
                ("sh_up", ctypes.c_void_p), ("sh_down", ctypes.c_void_p), ("down_gain", ctypes.c_void_p),
                ("down_gain2", ctypes.c_void_p), ("vq_codebook", ctypes.c_void_p), ("gate_plane", ctypes.c_void_p),
                ("up_plane", ctypes.c_void_p), ("down_plane", ctypes.c_void_p), ("gate_rowgain", ctypes.c_void_p),
                ("up_rowgain", ctypes.c_void_p), ("down_rowgain", ctypes.c_void_p)]


class Stats(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int32), ("path", ctypes.c_int32), ("n_unique", ctypes.c_int32),
                ("max_load", ctypes.c_int32), ("kernel_count", ctypes.c_int32)]


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int32), ("total_ms", ctypes.c_double)]


# Every symbol include/ds4moe.h declares: name -> (restype, argtypes)
_vp, _i32 = ctypes.c_void_p, ctypes.c_int32
SIGNATURES = {
    "ds4moe_create": (ctypes.c_int, [ctypes.POINTER(LayerDesc), ctypes.POINTER(Weights), ctypes.POINTER(_vp)]),
    "ds4moe_destroy": (ctypes.c_int, [_vp]),
    "ds4moe_set_stream": (ctypes.c_int, [_vp, _vp]),
    "ds4moe_route": (ctypes.c_int, [_vp, _vp, _i32, _vp, _vp]),
    "ds4moe_forward": (ctypes.c_int, [_vp, _vp, _i32, _vp]),
    "ds4moe_forward_host": (ctypes.c_int, [_vp, _vp, _i32, _vp]),
    "ds4moe_forward_path": (ctypes.c_int, [_vp, _vp, _i32, _i32, _vp]),
    "ds4moe_forward_routed": (ctypes.c_int, [_vp, _vp, _i32, _vp, _vp, _i32, _vp]),
    "ds4moe_route_detail": (ctypes.c_int, [_vp, _vp, _i32, _vp, _vp, _vp, _vp]),
    "ds4moe_status": (ctypes.c_int, [_vp]),
    "ds4moe_debug_skip_signal": (ctypes.c_int, [_vp, _i32]),
    "ds4moe_get_stats": (ctypes.c_int, [_vp, ctypes.POINTER(Stats)]),
    "ds4moe_inspect": (ctypes.c_int, [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.POINTER(_i32)]),
    "ds4moe_memory": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]),
    "ds4moe_profile": (ctypes.c_int, [_vp, _i32]),
    "ds4moe_profile_read": (ctypes.c_int, [_vp, ctypes.POINTER(KernelTime), _i32, ctypes.POINTER(_i32)]),
    "ds4moe_route_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp]),
    "ds4moe_strerror": (ctypes.c_char_p, [ctypes.c_int]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"ds4moe CUDA library not built ({LIB_PATH} missing); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


class DS4MoEError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {_lib.ds4moe_strerror(code).decode()} ({code})")


def _check(code: int, what: str):
    if code != DS4MOE_OK:
        raise DS4MoEError(code, what)


def _addr(t):
    """Device address of a torch tensor, or an int address, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


# ---- raw entry points (same names as the C ABI) ------------------------------

def ds4moe_create(desc: LayerDesc, weights: Weights) -> int:
    h = _vp()
    _check(_lib.ds4moe_create(ctypes.byref(desc), ctypes.byref(weights), ctypes.byref(h)), "ds4moe_create")
    return h.value


def ds4moe_destroy(h: int):
    _check(_lib.ds4moe_destroy(h), "ds4moe_destroy")


def ds4moe_set_stream(h: int, stream: int | None):
    _check(_lib.ds4moe_set_stream(h, stream or None), "ds4moe_set_stream")


def ds4moe_route(h: int, x, T: int, idx_out, w_out):
    _check(_lib.ds4moe_route(h, _addr(x), T, _addr(idx_out), _addr(w_out)), "ds4moe_route")


def ds4moe_route_detail(h: int, x, T: int, idx_out, w_out, gap_out=None, sel_out=None):
    _check(_lib.ds4moe_route_detail(h, _addr(x), T, _addr(idx_out), _addr(w_out), _addr(gap_out),
                                    _addr(sel_out)), "ds4moe_route_detail")


def ds4moe_forward(h: int, x, T: int, y):
    _check(_lib.ds4moe_forward(h, _addr(x), T, _addr(y)), "ds4moe_forward")


def ds4moe_forward_path(h: int, x, T: int, path: int, y):
    _check(_lib.ds4moe_forward_path(h, _addr(x), T, path, _addr(y)), "ds4moe_forward_path")


def ds4moe_forward_routed(h: int, x, T: int, idx, w, path: int, y):
    _check(_lib.ds4moe_forward_routed(h, _addr(x), T, _addr(idx), _addr(w), path, _addr(y)),
           "ds4moe_forward_routed")


def ds4moe_forward_host(h: int, x_host, T: int, y_host):
    _check(_lib.ds4moe_forward_host(h, _addr(x_host), T, _addr(y_host)), "ds4moe_forward_host")


def ds4moe_status(h: int) -> int:
    return int(_lib.ds4moe_status(h))


def ds4moe_debug_skip_signal(h: int, launches: int):
    _check(_lib.ds4moe_debug_skip_signal(h, launches), "ds4moe_debug_skip_signal")


def ds4moe_get_stats(h: int) -> Stats:
    s = Stats()
    _check(_lib.ds4moe_get_stats(h, ctypes.byref(s)), "ds4moe_get_stats")
    return s


def ds4moe_inspect(h: int, T: int, K: int, E: int, grouping: bool = True) -> dict:
    """Routing (and, with grouping, the expert grouping) of the last forward call, as numpy arrays."""
    import numpy as np
    idx = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float32)
    gap = np.empty((T,), dtype=np.float32)
    out = {"idx": idx, "w": w, "gap": gap}
    ptr = lambda a: a.ctypes.data if a is not None else None  # noqa: E731
    counts = inv = uexp = ustart = None
    nu = _i32()
    if grouping:
        counts = np.empty((E,), dtype=np.int32)
        inv = np.empty((T * K,), dtype=np.int32)
        uexp = np.empty((min(T * K, E),), dtype=np.int32)
        ustart = np.empty((min(T * K, E) + 1,), dtype=np.int32)
    _check(_lib.ds4moe_inspect(h, T, ptr(idx), ptr(w), ptr(gap), ptr(counts), ptr(inv), ptr(uexp), ptr(ustart),
                               ctypes.byref(nu) if grouping else None), "ds4moe_inspect")
    if grouping:
        n = nu.value
        out.update(counts=counts, inv=inv, uexp=uexp[:n].copy(), ustart=ustart[:n + 1].copy(), n_unique=n)
    return out


def ds4moe_memory(h: int):
    wb, sb = ctypes.c_uint64(), ctypes.c_uint64()
    _check(_lib.ds4moe_memory(h, ctypes.byref(wb), ctypes.byref(sb)), "ds4moe_memory")
    return wb.value, sb.value


def ds4moe_profile(h: int, enable: bool):
    _check(_lib.ds4moe_profile(h, 1 if enable else 0), "ds4moe_profile")


def ds4moe_profile_read(h: int) -> dict:
    """{kernel name: (launches, total_ms)} recorded since profiling was enabled."""
    buf = (KernelTime * 64)()
    n = _i32()
    _check(_lib.ds4moe_profile_read(h, buf, 64, ctypes.byref(n)), "ds4moe_profile_read")
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(min(n.value, 64))}


def ds4moe_route_noalloc(router_w, router_bias, x, T: int, H: int, E: int, K: int, idx_out, w_out,
                         stream=None):
    """Routing from the caller's router weights with no device allocation (fixed static scratch)."""
    _check(_lib.ds4moe_route_noalloc(_addr(router_w), _addr(router_bias), _addr(x), T, H, E, K, _addr(idx_out),
                                     _addr(w_out), stream or None), "ds4moe_route_noalloc")


def ds4moe_strerror(code: int) -> str:
    return _lib.ds4moe_strerror(code).decode()


def make_desc(hidden, inter, n_experts, top_k, shared_inter, max_tokens, flags=0) -> LayerDesc:
    return LayerDesc(DS4MOE_MAGIC, DS4MOE_VERSION, hidden, inter, n_experts, top_k, shared_inter, max_tokens,
                     flags)


# ---- convenience wrapper over torch tensors ----------------------------------

class MoELayer:
    """One ds4moe handle. Weights: dict of device torch tensors in the storage
    formats of ``include/ds4moe.h``, keyed by the ``ds4moe_weights`` field names
    (router_w, router_bias, gate, up, down, sh_gate, sh_up, sh_down, down_gain,
    down_gain2, and for VQ layers vq_codebook, *_plane, *_rowgain); optional
    ones may be None or absent."""

    def __init__(self, shape, weights: dict, max_tokens: int, flags: int = 0):
        self.shape = shape
        desc = make_desc(shape.hidden, shape.inter, shape.n_experts, shape.top_k, shape.shared_inter, max_tokens,
                         flags)
        w = Weights(*(_addr(weights.get(k)) for k, _ in Weights._fields_))
        self.handle = ds4moe_create(desc, w)
        self.max_tokens = max_tokens

    def close(self):
        if self.handle:
            ds4moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_stream(self, stream):
        ds4moe_set_stream(self.handle, stream.cuda_stream if hasattr(stream, "cuda_stream") else stream)

    def forward(self, x, y=None, path: int = PATH_AUTO):
        import torch
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.shape.hidden), dtype=torch.float32, device=x.device)
        ds4moe_forward_path(self.handle, x, T, path, y)
        return y

    def forward_routed(self, x, idx, w, y=None, path: int = PATH_AUTO):
        import torch
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.shape.hidden), dtype=torch.float32, device=x.device)
        ds4moe_forward_routed(self.handle, x, T, idx, w, path, y)
        return y

    def route(self, x, want_sel: bool = False):
        import torch
        T, K, E = x.shape[0], self.shape.top_k, self.shape.n_experts
        idx = torch.empty((T, K), dtype=torch.int32, device=x.device)
        w = torch.empty((T, K), dtype=torch.float32, device=x.device)
        gap = torch.empty((T,), dtype=torch.float32, device=x.device)
        sel = torch.empty((T, E), dtype=torch.float32, device=x.device) if want_sel else None
        ds4moe_route_detail(self.handle, x, T, idx, w, gap, sel)
        return idx, w, gap, sel

    def status(self) -> int:
        return ds4moe_status(self.handle)

    def stats(self) -> Stats:
        return ds4moe_get_stats(self.handle)

    def inspect(self, T: int, grouping: bool = True) -> dict:
        return ds4moe_inspect(self.handle, T, self.shape.top_k, self.shape.n_experts, grouping)
