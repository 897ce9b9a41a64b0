"""Seeded synthetic workloads for the routed-MoE layer.

This module draws inputs only; it contains none of the layer's arithmetic and
is shared by the CPU oracle tests, the GPU parity tests and the benchmark.
The C side (``ds4moe_synth.c``) does the drawing and the storage encodings.

Workloads (hidden H, routed intermediate I, experts E, top-k K, shared
intermediate I_sh, tokens T):

* ``tiny``          H=512,  I=256,  E=32,  K=6, I_sh=256,  T=4
* ``decode_t1``     H=4096, I=2048, E=384, K=6, I_sh=2048, T=1
* ``decode_t8``     the decode_t1 layer, T=8 tokens with independent seeds
* ``prefill_t1024`` the decode_t1 layer, T=1024 tokens, no router bias
* ``prefill_t4096_zipf4`` four independent layers shaped like decode_t1, each
  with a Zipf(s=1.1) rank profile added to the router's selection score,
  applied to the same T=4096 tokens.

Distributions: router ~ N(0, 0.02^2) fp32; 2-bit codes uniform 0..3, 4-bit
scales and mins uniform 0..15, d and dmin ~ |N(0, 0.01^2)| in binary16; 8-bit
codes uniform in [-127, 127] with d ~ |N(0, 0.001^2)|; x ~ N(0, 1) in bf16.
"""
from __future__ import annotations

import ctypes
import json
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ds4moe_synth.c")
_LIB = os.path.join(_HERE, "libds4moe_synth.so")

SEED_BASE = 0xD54E0000

# stream ids of the counter-based generator
S_ROUTER, S_GATE, S_UP, S_DOWN, S_SH_GATE, S_SH_UP, S_SH_DOWN, S_BIAS_RANK = range(1, 9)
S_GAIN1, S_GAIN2 = 9, 10
# VQ experts: codebook, then per matrix (gate, up, down) its bit plane and row gains
S_CODEBOOK = 11
S_GATE_PLANE, S_UP_PLANE, S_DOWN_PLANE = 12, 13, 14
S_GATE_ROWGAIN, S_UP_ROWGAIN, S_DOWN_ROWGAIN = 17, 18, 19
VQ_ROWGAIN_SIGMA = 0.05
GAIN_BLOCK_BYTES = 17
GAIN_SCALE_BYTE = 127 - 5  # E8M0 2^-5: gains 1 + 2^-5 * e2m1 in [0.8125, 1.1875]
MX4_BLOCK_BYTES = 17
MX4_SCALE_BYTE = 127 - 3  # MXFP4 weight scales 2^-3, 2^-4, 2^-5: |w| <= 0.75
S_X = 16

Q2_BLOCK_BYTES = 84
Q8_BLOCK_BYTES = 34

ZIPF_S = 1.1
ZIPF_BETA_FILE = os.path.join(_HERE, "zipf_beta.json")


def build(force: bool = False) -> str:
    """Compile the generator into a shared library next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.synth_fill_q2.argtypes = [u8p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double]
        lib.synth_fill_q8.argtypes = [u8p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double]
        lib.synth_fill_gain.argtypes = [u8p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint8]
        lib.synth_fill_mx4.argtypes = [u8p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint8]
        lib.synth_fill_bytes.argtypes = [u8p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_fill_e4m3_codebook.argtypes = [u8p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_fill_f16_abs_normal.argtypes = [ctypes.POINTER(ctypes.c_uint16), ctypes.c_int64, ctypes.c_uint64,
                                                  ctypes.c_uint64, ctypes.c_double]
        lib.synth_fill_normal_f32.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int64,
                                              ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double]
        lib.synth_fill_normal_bf16.argtypes = [ctypes.POINTER(ctypes.c_uint16), ctypes.c_int64,
                                               ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double]
        lib.synth_rank_permutation.argtypes = [ctypes.POINTER(ctypes.c_int32), ctypes.c_int32,
                                               ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_to_f16.argtypes = [ctypes.c_float]
        lib.synth_to_f16.restype = ctypes.c_uint16
        lib.synth_to_bf16.argtypes = [ctypes.c_float]
        lib.synth_to_bf16.restype = ctypes.c_uint16
        _lib = lib
    return _lib


def _ptr(a: np.ndarray, ct):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ct))


@dataclass(frozen=True)
class Shape:
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    shared_inter: int


@dataclass(frozen=True)
class Workload:
    name: str
    shape: Shape
    tokens: int
    n_layers: int
    zipf: bool
    layer_seeds: tuple
    description: str


TINY_SHAPE = Shape(512, 256, 32, 6, 256)
V4F_SHAPE = Shape(4096, 2048, 384, 6, 2048)

WORKLOADS = {
    "tiny": Workload("tiny", TINY_SHAPE, 4, 1, False, (SEED_BASE + 0,),
                     "tiny layer H=512 I=256 E=32 top-6 I_sh=256, T=4"),
    "decode_t1": Workload("decode_t1", V4F_SHAPE, 1, 1, False, (SEED_BASE + 1,),
                          "decode batch 1: H=4096 I=2048 E=384 top-6 I_sh=2048, T=1"),
    "decode_t8": Workload("decode_t8", V4F_SHAPE, 8, 1, False, (SEED_BASE + 1,),
                          "decode multi-session: the H=4096 E=384 layer, T=8 independent tokens"),
    "prefill_t1024": Workload("prefill_t1024", V4F_SHAPE, 1024, 1, False, (SEED_BASE + 1,),
                              "prefill chunk: the H=4096 E=384 layer, T=1024 tokens, near-uniform load"),
    "prefill_t4096_zipf4": Workload("prefill_t4096_zipf4", V4F_SHAPE, 4096, 4, True,
                                    tuple(SEED_BASE + 4 + 0x100 * l for l in range(4)),
                                    "long prefill with skew: 4 independent H=4096 E=384 layers, "
                                    "T=4096, Zipf(1.1) router bias (hottest ~20x mean load)"),
    # The decode <-> prefill crossover: the full layer with 64 tokens, each from its
    # own N(0,1) draw (~246 distinct experts, one to a few pairs each).
    "batch_t64": Workload("batch_t64", V4F_SHAPE, 64, 1, False, (SEED_BASE + 1,),
                          "verify/multi-session batch: the H=4096 E=384 layer, T=64 tokens"),
    # The same token count on 48 experts (~8 pairs per expert, <1 GB on the device)
    # for profiler captures of the batch kernels.
    "batch_profile": Workload("batch_profile", Shape(4096, 2048, 48, 6, 2048), 64, 1, False, (SEED_BASE + 9,),
                              "profiling case: H=4096 I=2048 E=48 top-6 I_sh=2048, T=64"),
    # A reduced copy of the prefill layer for profiler captures: the same expert
    # matrices (H=4096, I=2048) but 48 experts (~400 MB of 2-bit rows, above the
    # L2 size) and 128 tokens, so one launch is short.
    "prefill_profile": Workload("prefill_profile", Shape(4096, 2048, 48, 6, 2048), 128, 1, False,
                                (SEED_BASE + 5,),
                                "profiling case: H=4096 I=2048 E=48 top-6 I_sh=2048, T=128"),
    # The same for the decode kernel: one token, the full-size expert matrices,
    # 48 experts, so a full profiler capture holds ~0.8 GB on the device.
    "decode_profile": Workload("decode_profile", Shape(4096, 2048, 48, 6, 2048), 1, 1, False,
                               (SEED_BASE + 7,),
                               "profiling case: H=4096 I=2048 E=48 top-6 I_sh=2048, T=1"),
    # Hot experts for the tensor-bound regime of the skewed prefill (whose
    # hottest experts take ~1,280 tokens): 8 experts, 1024 tokens, ~768 tokens
    # per expert; ~0.2 GB of expert rows, so a full capture stays small.
    "prefill_hot_profile": Workload("prefill_hot_profile", Shape(4096, 2048, 8, 6, 2048), 1024, 1, False,
                                    (SEED_BASE + 8,),
                                    "profiling case: H=4096 I=2048 E=8 top-6 I_sh=2048, T=1024 (~768 tokens per expert)"),
}


def q2_matrix(rows: int, k: int, seed: int, stream: int, sigma: float = 0.01) -> np.ndarray:
    assert k % 256 == 0
    out = np.empty((rows, k // 256, Q2_BLOCK_BYTES), dtype=np.uint8)
    _load().synth_fill_q2(_ptr(out, ctypes.c_uint8), out.shape[0] * out.shape[1], seed, stream, sigma)
    return out


def q8_matrix(rows: int, k: int, seed: int, stream: int, sigma: float = 0.001) -> np.ndarray:
    assert k % 32 == 0
    out = np.empty((rows, k // 32, Q8_BLOCK_BYTES), dtype=np.uint8)
    _load().synth_fill_q8(_ptr(out, ctypes.c_uint8), out.shape[0] * out.shape[1], seed, stream, sigma)
    return out


def normal_f32(n: int, seed: int, stream: int, sigma: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().synth_fill_normal_f32(_ptr(out, ctypes.c_float), n, seed, stream, sigma)
    return out


def normal_bf16(n: int, seed: int, stream: int, sigma: float = 1.0) -> np.ndarray:
    """Raw bfloat16 bits (uint16)."""
    out = np.empty(n, dtype=np.uint16)
    _load().synth_fill_normal_bf16(_ptr(out, ctypes.c_uint16), n, seed, stream, sigma)
    return out


def rank_permutation(n: int, seed: int, stream: int = S_BIAS_RANK) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().synth_rank_permutation(_ptr(out, ctypes.c_int32), n, seed, stream)
    return out


def f32_to_f16_bits(v: float) -> int:
    return int(_load().synth_to_f16(v))


def f32_to_bf16_bits(v: float) -> int:
    return int(_load().synth_to_bf16(v))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Decode raw bfloat16 bits (a plain bit shift; used to hand activations to tests)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def zipf_profile(n_experts: int, layer_seed: int) -> np.ndarray:
    """r_e^-s for a seeded rank permutation r (rank 1 = hottest expert)."""
    ranks = rank_permutation(n_experts, layer_seed).astype(np.float64)
    return ranks ** (-ZIPF_S)


def zipf_beta(layer_seed: int) -> float:
    """Bias magnitude for one skewed layer, read from the committed calibration file."""
    with open(ZIPF_BETA_FILE) as f:
        table = json.load(f)
    return float(table["beta"][str(layer_seed)])


def gain_table(n_experts: int, hidden: int, seed: int, stream: int, scale_byte: int = GAIN_SCALE_BYTE) -> np.ndarray:
    """Per-expert down gains: [E][H/32] blocks of 17 bytes (FP4 codes, E8M0 scale)."""
    n = n_experts * (hidden // 32)
    out = np.empty(n * GAIN_BLOCK_BYTES, dtype=np.uint8)
    _load().synth_fill_gain(_ptr(out, ctypes.c_uint8), n, seed, stream, scale_byte)
    return out.reshape(n_experts, hidden // 32, GAIN_BLOCK_BYTES)


def mx4_matrix(rows: int, k: int, seed: int, stream: int, base_byte: int = MX4_SCALE_BYTE) -> np.ndarray:
    """MXFP4 weights [rows][k/32] blocks of 17 bytes."""
    assert k % 32 == 0
    out = np.empty((rows, k // 32, MX4_BLOCK_BYTES), dtype=np.uint8)
    _load().synth_fill_mx4(_ptr(out, ctypes.c_uint8), out.shape[0] * out.shape[1], seed, stream, base_byte)
    return out


def random_bytes(n: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    _load().synth_fill_bytes(_ptr(out, ctypes.c_uint8), n, seed, stream)
    return out


def e4m3_codebook(entries: int, seed: int, stream: int = S_CODEBOOK) -> np.ndarray:
    """[entries][8] FP8 E4M3 codeword bytes."""
    out = np.empty(entries * 8, dtype=np.uint8)
    _load().synth_fill_e4m3_codebook(_ptr(out, ctypes.c_uint8), out.size, seed, stream)
    return out.reshape(entries, 8)


def f16_abs_normal(n: int, seed: int, stream: int, sigma: float) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    _load().synth_fill_f16_abs_normal(_ptr(out, ctypes.c_uint16), n, seed, stream, sigma)
    return out


def vq_matrix(n_experts: int, rows: int, k: int, bits: int, seed: int, stream: int, plane_stream: int,
              gain_stream: int):
    """One VQ matrix: (index streams [E][rows*k/8*3/2] bytes, bit planes [E][rows*k/64] or
    None, row gains [E][rows] binary16 bits). Indices are uniform."""
    n = rows * (k // 8)
    idx = random_bytes(n_experts * n * 3 // 2, seed, stream).reshape(n_experts, n * 3 // 2)
    plane = random_bytes(n_experts * n // 8, seed, plane_stream).reshape(n_experts, n // 8) if bits == 13 else None
    g = f16_abs_normal(n_experts * rows, seed, gain_stream, VQ_ROWGAIN_SIGMA).reshape(n_experts, rows)
    return idx, plane, g


def make_layer(shape: Shape, seed: int, zipf: bool = False, zipf_beta_value: float | None = None,
               gains: int = 0, routed_format: str = "q2", vq_bits: int = 12) -> dict:
    """All weights of one layer in canonical layout (host numpy arrays).

    gains: number of down-gain tables to draw (0, 1 or 2) as "down_gain", "down_gain2".
    routed_format: "q2" (2-bit blocks), "mx4" (MXFP4 blocks, same streams) or "vq"
    (vq_bits-bit indices into one E4M3 codebook, with row gains)."""
    H, I, E, Ish = shape.hidden, shape.inter, shape.n_experts, shape.shared_inter
    layer = {"router_w": normal_f32(E * H, seed, S_ROUTER, 0.02).reshape(E, H), "router_bias": None}
    if routed_format == "q2":
        layer["gate"] = q2_matrix(E * I, H, seed, S_GATE).reshape(E, I, H // 256, Q2_BLOCK_BYTES)
        layer["up"] = q2_matrix(E * I, H, seed, S_UP).reshape(E, I, H // 256, Q2_BLOCK_BYTES)
        layer["down"] = q2_matrix(E * H, I, seed, S_DOWN).reshape(E, H, I // 256, Q2_BLOCK_BYTES)
    elif routed_format == "mx4":
        layer["gate"] = mx4_matrix(E * I, H, seed, S_GATE).reshape(E, I, H // 32, MX4_BLOCK_BYTES)
        layer["up"] = mx4_matrix(E * I, H, seed, S_UP).reshape(E, I, H // 32, MX4_BLOCK_BYTES)
        layer["down"] = mx4_matrix(E * H, I, seed, S_DOWN).reshape(E, H, I // 32, MX4_BLOCK_BYTES)
        layer["routed_format"] = "mx4"
    elif routed_format == "vq":
        assert vq_bits in (12, 13)
        layer["routed_format"] = "vq"
        layer["vq_bits"] = vq_bits
        layer["vq_codebook"] = e4m3_codebook(1 << vq_bits, seed)
        for name, rows, k, s_idx, s_plane, s_gain in (("gate", I, H, S_GATE, S_GATE_PLANE, S_GATE_ROWGAIN),
                                                      ("up", I, H, S_UP, S_UP_PLANE, S_UP_ROWGAIN),
                                                      ("down", H, I, S_DOWN, S_DOWN_PLANE, S_DOWN_ROWGAIN)):
            layer[name], layer[name + "_plane"], layer[name + "_rowgain"] = vq_matrix(
                E, rows, k, vq_bits, seed, s_idx, s_plane, s_gain)
    else:
        raise ValueError(routed_format)
    if Ish > 0:
        layer["sh_gate"] = q8_matrix(Ish, H, seed, S_SH_GATE)
        layer["sh_up"] = q8_matrix(Ish, H, seed, S_SH_UP)
        layer["sh_down"] = q8_matrix(H, Ish, seed, S_SH_DOWN)
    else:
        layer["sh_gate"] = layer["sh_up"] = layer["sh_down"] = None
    if zipf:
        beta = zipf_beta(seed) if zipf_beta_value is None else zipf_beta_value
        layer["router_bias"] = (beta * zipf_profile(E, seed)).astype(np.float32)
    if gains >= 1:
        layer["down_gain"] = gain_table(E, H, seed, S_GAIN1)
    if gains >= 2:
        layer["down_gain2"] = gain_table(E, H, seed, S_GAIN2)
    return layer


def token_seed(workload: str, t: int) -> int:
    """Seed of token t for the decode workloads (one seed per token)."""
    if workload == "decode_t1":
        return SEED_BASE + 1 + 0x20000 + t
    if workload == "decode_t8":
        return SEED_BASE + 2 + 0x10000 + t
    raise KeyError(workload)


def make_tokens(workload: str, T: int | None = None, first: int = 0) -> np.ndarray:
    """bf16 activations [T, H] (raw bits) of a workload.

    Decode workloads draw each token from its own seed; ``first`` offsets the
    token index, which gives the rotating token pool used for timing.
    """
    wl = WORKLOADS[workload]
    H = wl.shape.hidden
    T = wl.tokens if T is None else T
    if workload in ("decode_t1", "decode_t8"):
        return np.stack([normal_bf16(H, token_seed(workload, first + t), S_X) for t in range(T)])
    if workload == "tiny":
        return normal_bf16(T * H, SEED_BASE + 0 + 0x10000, S_X).reshape(T, H)
    if workload == "prefill_t1024":
        return normal_bf16(T * H, SEED_BASE + 3, S_X).reshape(T, H)
    if workload == "prefill_t4096_zipf4":
        return normal_bf16(T * H, SEED_BASE + 4 + 0x10000, S_X).reshape(T, H)
    if workload == "prefill_profile":
        return normal_bf16(T * H, SEED_BASE + 5 + 0x10000, S_X).reshape(T, H)
    if workload == "decode_profile":
        return normal_bf16(T * H, SEED_BASE + 7 + 0x10000, S_X).reshape(T, H)
    if workload == "batch_t64":
        return normal_bf16(T * H, SEED_BASE + 0x100 + T, S_X).reshape(T, H)
    if workload == "batch_profile":
        return normal_bf16(T * H, SEED_BASE + 9 + 0x10000, S_X).reshape(T, H)
    if workload == "prefill_hot_profile":
        return normal_bf16(T * H, SEED_BASE + 8 + 0x10000, S_X).reshape(T, H)
    raise KeyError(workload)
