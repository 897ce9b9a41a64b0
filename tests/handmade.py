"""Hand-built layers whose outputs have closed forms.

The encoder here writes the storage layout from its field definition (2-bit
block: scales[16] with the scale in the low nibble and the min in the high
nibble, 64 bytes of LSB-first 2-bit codes, binary16 d, binary16 dmin; 8-bit
block: binary16 d then 32 int8 codes). binary16 bit patterns come from numpy's
own float16 conversion, which is independent of both the oracle and the
generator.
"""
import numpy as np


def f16_bits(v: float) -> int:
    return int(np.array([v], dtype=np.float16).view(np.uint16)[0])


def q2_block(d: float, dmin: float, sc, m, q) -> bytes:
    sc = np.broadcast_to(np.asarray(sc, dtype=np.int64), (16,))
    m = np.broadcast_to(np.asarray(m, dtype=np.int64), (16,))
    q = np.broadcast_to(np.asarray(q, dtype=np.int64), (256,))
    assert ((0 <= sc) & (sc < 16)).all() and ((0 <= m) & (m < 16)).all() and ((0 <= q) & (q < 4)).all()
    scales = bytes(int(sc[j]) | (int(m[j]) << 4) for j in range(16))
    qs = bytes(sum(int(q[4 * b + s]) << (2 * s) for s in range(4)) for b in range(64))
    return scales + qs + f16_bits(d).to_bytes(2, "little") + f16_bits(dmin).to_bytes(2, "little")


def q8_block(d: float, q) -> bytes:
    q = np.broadcast_to(np.asarray(q, dtype=np.int64), (32,))
    assert ((-128 <= q) & (q < 128)).all()
    return f16_bits(d).to_bytes(2, "little") + bytes(int(v) & 0xFF for v in q)


def as_u8(blocks_2d) -> np.ndarray:
    """list (rows) of lists (blocks) of bytes -> uint8 [rows, nblocks, block_bytes]."""
    rows = [b"".join(r) for r in blocks_2d]
    nb = len(blocks_2d[0])
    return np.frombuffer(b"".join(rows), dtype=np.uint8).reshape(len(rows), nb, -1).copy()


def bf16_bits(v) -> np.ndarray:
    """float32 values that are exact in bf16 -> raw bits."""
    a = np.asarray(v, dtype=np.float32)
    bits = a.view(np.uint32)
    assert (bits & 0xFFFF == 0).all(), "value not exact in bf16"
    return (bits >> 16).astype(np.uint16)


def gain_block(codes, scale_byte: int) -> bytes:
    """Down-gain block: 32 four-bit E2M1 codes, channel i in byte i // 2 with the
    even channel in the low nibble, then the E8M0 scale byte."""
    c = np.broadcast_to(np.asarray(codes, dtype=np.int64), (32,))
    assert ((0 <= c) & (c < 16)).all() and 0 <= scale_byte < 256
    return bytes(int(c[2 * b]) | (int(c[2 * b + 1]) << 4) for b in range(16)) + bytes([scale_byte])
