"""ctypes wrapper of the CPU oracle (``ds4moe_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this module; the product path never does. It
shares no code with the CUDA library and imports nothing from it.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ds4moe_oracle.c")
_LIB = os.path.join(_HERE, "libds4moe_oracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle (plain C, OpenMP, no fused multiply-add contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                               "-std=c11", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Shape(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("shared_inter", ctypes.c_int32)]


_lib = None
_vp = ctypes.c_void_p


class _VqMat(ctypes.Structure):
    _fields_ = [("stream", ctypes.c_void_p), ("plane", ctypes.c_void_p), ("gains", ctypes.c_void_p)]


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Temporarily route every call through another build of the oracle (tests only)."""
    global _lib
    saved = _lib
    _lib = _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def _configure(lib):
    lib.oracle_f16.argtypes = [ctypes.c_uint16]
    lib.oracle_f16.restype = ctypes.c_double
    lib.oracle_bf16.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16.restype = ctypes.c_double
    lib.oracle_silu.argtypes = [ctypes.c_double]
    lib.oracle_silu.restype = ctypes.c_double
    lib.oracle_sigmoid.argtypes = [ctypes.c_double]
    lib.oracle_sigmoid.restype = ctypes.c_double
    lib.oracle_max_threads.restype = ctypes.c_int32
    lib.oracle_dequant_q2.argtypes = [_vp, _vp]
    lib.oracle_dequant_q8.argtypes = [_vp, _vp]
    lib.oracle_dequant_q2_row.argtypes = [_vp, ctypes.c_int64, _vp]
    lib.oracle_dequant_q8_row.argtypes = [_vp, ctypes.c_int64, _vp]
    lib.oracle_route.argtypes = [ctypes.POINTER(_Shape), _vp, _vp, _vp, ctypes.c_int32,
                                 _vp, _vp, _vp, _vp, _vp]
    lib.oracle_route.restype = ctypes.c_int
    lib.oracle_logits.argtypes = [ctypes.POINTER(_Shape), _vp, _vp, ctypes.c_int32, _vp]
    lib.oracle_logits.restype = ctypes.c_int
    lib.oracle_select.argtypes = [ctypes.POINTER(_Shape), _vp, _vp, ctypes.c_int32, _vp, _vp, _vp, _vp]
    lib.oracle_select.restype = ctypes.c_int
    lib.oracle_expert_q2.argtypes = [ctypes.POINTER(_Shape), _vp, _vp, _vp, _vp, _vp]
    lib.oracle_shared_q8.argtypes = [ctypes.POINTER(_Shape), _vp, _vp, _vp, _vp, _vp]
    lib.oracle_e2m1.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1.restype = ctypes.c_double
    lib.oracle_e8m0.argtypes = [ctypes.c_uint8]
    lib.oracle_e8m0.restype = ctypes.c_double
    lib.oracle_gain_block.argtypes = [_vp, _vp]
    lib.oracle_dequant_mx4.argtypes = [_vp, _vp]
    lib.oracle_e4m3.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3.restype = ctypes.c_double
    lib.oracle_vq_index.argtypes = [_vp, _vp, ctypes.c_int64]
    lib.oracle_vq_index.restype = ctypes.c_int32
    lib.oracle_dequant_vq_row.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int64, ctypes.c_int64, _vp]
    lib.oracle_expert_vq.argtypes = [ctypes.POINTER(_Shape), _vp, ctypes.POINTER(_VqMat), ctypes.POINTER(_VqMat),
                                     ctypes.POINTER(_VqMat), ctypes.c_int32, _vp, _vp]
    lib.oracle_forward_routed_vq.argtypes = [ctypes.POINTER(_Shape), _vp, ctypes.POINTER(_VqMat),
                                             ctypes.POINTER(_VqMat), ctypes.POINTER(_VqMat), _vp, _vp, _vp, _vp, _vp,
                                             _vp, ctypes.c_int32, _vp, _vp, _vp, ctypes.c_int32]
    lib.oracle_forward_routed_vq.restype = ctypes.c_int
    lib.oracle_act_q8.argtypes = [_vp, ctypes.c_int64, _vp, _vp]
    lib.oracle_act_mx4.argtypes = [_vp, ctypes.c_int64, _vp, _vp]
    lib.oracle_e2m1_nearest.argtypes = [ctypes.c_double]
    lib.oracle_e2m1_nearest.restype = ctypes.c_uint8
    lib.oracle_expert_mx4.argtypes = [ctypes.POINTER(_Shape), ctypes.c_int32, _vp, _vp, _vp, _vp, _vp]
    lib.oracle_forward_routed_mx4.argtypes = [ctypes.POINTER(_Shape), ctypes.c_int32, _vp, _vp, _vp, _vp, _vp, _vp,
                                              _vp, _vp, _vp, ctypes.c_int32, _vp, _vp, _vp, ctypes.c_int32]
    lib.oracle_forward_routed_mx4.restype = ctypes.c_int
    lib.oracle_forward_routed_gain.argtypes = [ctypes.POINTER(_Shape), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                               _vp, ctypes.c_int32, _vp, _vp, _vp, ctypes.c_int32]
    lib.oracle_forward_routed_gain.restype = ctypes.c_int
    lib.oracle_forward_routed.argtypes = [ctypes.POINTER(_Shape), _vp, _vp, _vp, _vp, _vp, _vp,
                                          _vp, ctypes.c_int32, _vp, _vp, _vp, ctypes.c_int32]
    lib.oracle_forward_routed.restype = ctypes.c_int
    return lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _shape(shape) -> _Shape:
    return _Shape(shape.hidden, shape.inter, shape.n_experts, shape.top_k, shape.shared_inter)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def f16(bits: int) -> float:
    return float(_load().oracle_f16(bits))


def bf16(bits: int) -> float:
    return float(_load().oracle_bf16(bits))


def silu(z: float) -> float:
    return float(_load().oracle_silu(z))


def sigmoid(z: float) -> float:
    return float(_load().oracle_sigmoid(z))


def dequant_q2(block: np.ndarray) -> np.ndarray:
    """84-byte block -> 256 float64 weights."""
    b = np.ascontiguousarray(block, dtype=np.uint8).reshape(84)
    out = np.empty(256, dtype=np.float64)
    _load().oracle_dequant_q2(_p(b), _p(out))
    return out


def dequant_q8(block: np.ndarray) -> np.ndarray:
    """34-byte block -> 32 float64 weights."""
    b = np.ascontiguousarray(block, dtype=np.uint8).reshape(34)
    out = np.empty(32, dtype=np.float64)
    _load().oracle_dequant_q8(_p(b), _p(out))
    return out


def dequant_q2_matrix(m: np.ndarray) -> np.ndarray:
    """[rows, nblocks, 84] -> [rows, 256*nblocks] float64."""
    m = np.ascontiguousarray(m, dtype=np.uint8)
    rows, nb = m.shape[0], m.shape[1]
    out = np.empty((rows, nb * 256), dtype=np.float64)
    for r in range(rows):
        _load().oracle_dequant_q2_row(m[r].ctypes.data, nb * 256, out[r].ctypes.data)
    return out


def dequant_q8_matrix(m: np.ndarray) -> np.ndarray:
    m = np.ascontiguousarray(m, dtype=np.uint8)
    rows, nb = m.shape[0], m.shape[1]
    out = np.empty((rows, nb * 32), dtype=np.float64)
    for r in range(rows):
        _load().oracle_dequant_q8_row(m[r].ctypes.data, nb * 32, out[r].ctypes.data)
    return out


def route(shape, router_w: np.ndarray, router_bias, x_bf16: np.ndarray, want_logits: bool = False):
    """Returns dict(idx [T,K] int32, weights [T,K] f64, gap [T] f64, sel [T,E] f32, logits?)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T = x.shape[0]
    E, K = shape.n_experts, shape.top_k
    rw = np.ascontiguousarray(router_w, dtype=np.float32)
    rb = None if router_bias is None else np.ascontiguousarray(router_bias, dtype=np.float32)
    idx = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    gap = np.empty(T, dtype=np.float64)
    sel = np.empty((T, E), dtype=np.float32)
    logits = np.empty((T, E), dtype=np.float64) if want_logits else None
    s = _shape(shape)
    rc = _load().oracle_route(ctypes.byref(s), _p(rw), _p(rb), _p(x), T, _p(idx), _p(w), _p(gap),
                              _p(logits), _p(sel))
    if rc != 0:
        raise ValueError("oracle_route rejected the shape")
    out = {"idx": idx, "weights": w, "gap": gap, "sel": sel}
    if want_logits:
        out["logits"] = logits
    return out


def logits(shape, router_w: np.ndarray, x_bf16: np.ndarray) -> np.ndarray:
    """Exact router logits [T, E] float64."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rw = np.ascontiguousarray(router_w, dtype=np.float32)
    out = np.empty((x.shape[0], shape.n_experts), dtype=np.float64)
    s = _shape(shape)
    if _load().oracle_logits(ctypes.byref(s), _p(rw), _p(x), x.shape[0], _p(out)) != 0:
        raise ValueError("oracle_logits rejected the shape")
    return out


def select(shape, logits_tE: np.ndarray, router_bias):
    """Selection from given logits: dict(idx, weights, gap, sel)."""
    L = np.ascontiguousarray(logits_tE, dtype=np.float64)
    T, E, K = L.shape[0], shape.n_experts, shape.top_k
    rb = None if router_bias is None else np.ascontiguousarray(router_bias, dtype=np.float32)
    idx = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    gap = np.empty(T, dtype=np.float64)
    sel = np.empty((T, E), dtype=np.float32)
    s = _shape(shape)
    if _load().oracle_select(ctypes.byref(s), _p(L), _p(rb), T, _p(idx), _p(w), _p(gap), _p(sel)) != 0:
        raise ValueError("oracle_select rejected the shape")
    return {"idx": idx, "weights": w, "gap": gap, "sel": sel}


def e2m1(code: int) -> float:
    """Value of a 4-bit FP4 E2M1 code."""
    return _load().oracle_e2m1(code)


def e8m0(x: int) -> float:
    """Value of an E8M0 block scale byte, 2^(x - 127)."""
    return _load().oracle_e8m0(x)


def gain_block(block: np.ndarray) -> np.ndarray:
    """The 32 down gains of one 17-byte gain block."""
    b = np.ascontiguousarray(block, dtype=np.uint8)
    assert b.size == 17
    s = np.empty(32, dtype=np.float64)
    _load().oracle_gain_block(_p(b), _p(s))
    return s


ACT = {"exact": 0, "q8": 1, "mx4": 2}


def dequant_mx4(block: np.ndarray) -> np.ndarray:
    """The 32 weights of one 17-byte MXFP4 block."""
    b = np.ascontiguousarray(block, dtype=np.uint8)
    assert b.size == 17
    w = np.empty(32, dtype=np.float64)
    _load().oracle_dequant_mx4(_p(b), _p(w))
    return w


def act_q8(x_f32: np.ndarray):
    """Q8 activation blocks of a float32 vector: (d float32 [n/32], q int8 [n])."""
    x = np.ascontiguousarray(x_f32, dtype=np.float32)
    d = np.empty(x.size // 32, dtype=np.float32)
    q = np.empty(x.size, dtype=np.int8)
    _load().oracle_act_q8(_p(x), x.size, _p(d), _p(q))
    return d, q


def act_mx4(x_f32: np.ndarray):
    """MXFP4 activation blocks of a float32 vector: (E8M0 bytes [n/32], E2M1 codes [n])."""
    x = np.ascontiguousarray(x_f32, dtype=np.float32)
    sc = np.empty(x.size // 32, dtype=np.uint8)
    c = np.empty(x.size, dtype=np.uint8)
    _load().oracle_act_mx4(_p(x), x.size, _p(sc), _p(c))
    return sc, c


def e2m1_nearest(r: float) -> int:
    return int(_load().oracle_e2m1_nearest(r))


def expert_mx4(shape, act: str, gate_e: np.ndarray, up_e: np.ndarray, down_e: np.ndarray,
               xt: np.ndarray) -> np.ndarray:
    """One MXFP4 routed expert on one float64 activation vector, activations quantised by act."""
    xt = np.ascontiguousarray(xt, dtype=np.float64)
    ye = np.empty(shape.hidden, dtype=np.float64)
    s = _shape(shape)
    g, u, d = (np.ascontiguousarray(a, dtype=np.uint8) for a in (gate_e, up_e, down_e))
    _load().oracle_expert_mx4(ctypes.byref(s), ACT[act], _p(g), _p(u), _p(d), _p(xt), _p(ye))
    return ye


def e4m3(b: int) -> float:
    """Value of an FP8 E4M3 byte."""
    return _load().oracle_e4m3(b)


def vq_index(stream: np.ndarray, plane, k: int) -> int:
    """Index k of a VQ index stream (with bit 12 from the plane, if given)."""
    st = np.ascontiguousarray(stream, dtype=np.uint8)
    pl = None if plane is None else np.ascontiguousarray(plane, dtype=np.uint8)
    return int(_load().oracle_vq_index(_p(st), _p(pl), k))


def dequant_vq_row(codebook, stream, plane, gains, r: int, k: int) -> np.ndarray:
    """Row r (k weights) of one expert's VQ matrix."""
    cb = np.ascontiguousarray(codebook, dtype=np.uint8)
    st = np.ascontiguousarray(stream, dtype=np.uint8)
    pl = None if plane is None else np.ascontiguousarray(plane, dtype=np.uint8)
    g = np.ascontiguousarray(gains, dtype=np.uint16)
    w = np.empty(k, dtype=np.float64)
    _load().oracle_dequant_vq_row(_p(cb), _p(st), _p(pl), _p(g), r, k, _p(w))
    return w


def _vq_mats(layer):
    keep = []
    mats = []
    for name in ("gate", "up", "down"):
        arrs = [np.ascontiguousarray(layer[name], dtype=np.uint8),
                None if layer.get(name + "_plane") is None else np.ascontiguousarray(layer[name + "_plane"],
                                                                                     dtype=np.uint8),
                np.ascontiguousarray(layer[name + "_rowgain"], dtype=np.uint16)]
        keep += arrs
        mats.append(_VqMat(*(_p(a) for a in arrs)))
    return mats, keep


def expert_vq(shape, layer: dict, e: int, xt: np.ndarray) -> np.ndarray:
    """VQ routed expert e of the layer on one float64 activation vector."""
    xt = np.ascontiguousarray(xt, dtype=np.float64)
    ye = np.empty(shape.hidden, dtype=np.float64)
    s = _shape(shape)
    mats, keep = _vq_mats(layer)
    cb = np.ascontiguousarray(layer["vq_codebook"], dtype=np.uint8)
    _load().oracle_expert_vq(ctypes.byref(s), _p(cb), *(ctypes.byref(m) for m in mats), e, _p(xt), _p(ye))
    return ye


def forward_routed(shape, layer: dict, x_bf16: np.ndarray, idx: np.ndarray, weights: np.ndarray,
                   nthreads: int = 0, act: str | None = None) -> np.ndarray:
    """Layer output [T, H] float64 for the given routing (with the layer's down gains
    "down_gain" / "down_gain2", where present). A layer whose "routed_format" is
    "mx4" needs act: the activation quantisation of its expert products ("q8"
    decode, "mx4" prefill, "exact")."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T = x.shape[0]
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    weights = np.ascontiguousarray(weights, dtype=np.float64)
    y = np.empty((T, shape.hidden), dtype=np.float64)
    s = _shape(shape)
    common = (_p(layer["gate"]), _p(layer["up"]), _p(layer["down"]), _p(layer.get("sh_gate")),
              _p(layer.get("sh_up")), _p(layer.get("sh_down")), _p(layer.get("down_gain")),
              _p(layer.get("down_gain2")), _p(x), T, _p(idx), _p(weights), _p(y), nthreads)
    if layer.get("routed_format", "q2") == "vq":
        mats, keep = _vq_mats(layer)
        cb = np.ascontiguousarray(layer["vq_codebook"], dtype=np.uint8)
        rc = _load().oracle_forward_routed_vq(ctypes.byref(s), _p(cb), *(ctypes.byref(m) for m in mats),
                                              *common[3:])
    elif layer.get("routed_format", "q2") == "mx4":
        rc = _load().oracle_forward_routed_mx4(ctypes.byref(s), ACT[act], *common)
    else:
        assert act in (None, "exact"), "2-bit routed experts take exact activations"
        rc = _load().oracle_forward_routed_gain(ctypes.byref(s), *common)
    if rc != 0:
        raise ValueError("oracle_forward_routed rejected its arguments")
    return y


def forward(shape, layer: dict, x_bf16: np.ndarray, nthreads: int = 0, act: str | None = None):
    """Route, then compute the layer. Returns (y [T,H] f64, routing dict)."""
    r = route(shape, layer["router_w"], layer.get("router_bias"), x_bf16)
    y = forward_routed(shape, layer, x_bf16, r["idx"], r["weights"], nthreads, act)
    return y, r


def expert(shape, gate_e: np.ndarray, up_e: np.ndarray, down_e: np.ndarray, xt: np.ndarray) -> np.ndarray:
    """One routed expert on one float64 activation vector."""
    xt = np.ascontiguousarray(xt, dtype=np.float64)
    ye = np.empty(shape.hidden, dtype=np.float64)
    s = _shape(shape)
    g, u, d = (np.ascontiguousarray(a, dtype=np.uint8) for a in (gate_e, up_e, down_e))
    _load().oracle_expert_q2(ctypes.byref(s), _p(g), _p(u), _p(d), _p(xt), _p(ye))
    return ye


def shared(shape, sh_gate: np.ndarray, sh_up: np.ndarray, sh_down: np.ndarray, xt: np.ndarray) -> np.ndarray:
    xt = np.ascontiguousarray(xt, dtype=np.float64)
    ysh = np.empty(shape.hidden, dtype=np.float64)
    s = _shape(shape)
    g, u, d = (np.ascontiguousarray(a, dtype=np.uint8) for a in (sh_gate, sh_up, sh_down))
    _load().oracle_shared_q8(ctypes.byref(s), _p(g), _p(u), _p(d), _p(xt), _p(ysh))
    return ysh
