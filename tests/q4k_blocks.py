"""Test-side construction of Q4_K blocks with known contents.

Written from the format description, independently of both the oracle and the
CUDA library: 144 bytes per 256 weights = fp16 d (bytes 0-1), fp16 dmin
(bytes 2-3), 12 bytes of packed 6-bit (scale, min) pairs for the eight
32-weight sub-blocks (bytes 4-15), 128 bytes of 4-bit codes (bytes 16-143),
and w = d*sc*q - dmin*m.

Scale packing table (byte index into the 12 scale bytes):
  sub-block j in 0..3: scale bits 0-5 -> byte j bits 0-5; min bits 0-5 -> byte j+4 bits 0-5
  sub-block j in 4..7: scale bits 0-3 -> byte j+4 bits 0-3; scale bits 4-5 -> byte j-4 bits 6-7
                       min bits 0-3   -> byte j+4 bits 4-7; min bits 4-5   -> byte j bits 6-7
Code packing: weight 64g+l (l < 32) is the low nibble of code byte 32g+l, weight
64g+32+l its high nibble.
"""
import numpy as np


def f16_bits(v: float) -> int:
    return int(np.array([v], dtype=np.float16).view(np.uint16)[0])


def pack_scales(sc, m) -> bytes:
    b = [0] * 12
    for j in range(8):
        s, mm = int(sc[j]), int(m[j])
        assert 0 <= s < 64 and 0 <= mm < 64
        if j < 4:
            b[j] |= s
            b[j + 4] |= mm
        else:
            b[j + 4] |= (s & 0xF) | ((mm & 0xF) << 4)
            b[j - 4] |= (s >> 4) << 6
            b[j] |= (mm >> 4) << 6
    return bytes(b)


def pack_codes(q) -> bytes:
    q = [int(v) for v in q]
    assert len(q) == 256 and all(0 <= v < 16 for v in q)
    out = bytearray(128)
    for g in range(4):
        for l in range(32):
            out[32 * g + l] = q[64 * g + l] | (q[64 * g + 32 + l] << 4)
    return bytes(out)


def make_block(d: float, dmin: float, sc, m, q) -> bytes:
    db, mb = f16_bits(d), f16_bits(dmin)
    head = bytes([db & 0xFF, db >> 8, mb & 0xFF, mb >> 8])
    return head + pack_scales(sc, m) + pack_codes(q)


def block_values(d: float, dmin: float, sc, m, q) -> np.ndarray:
    """Exact dequantised values (float64 arithmetic, then one rounding to fp32)."""
    d64 = float(np.float16(d))
    m64 = float(np.float16(dmin))
    out = np.empty(256, dtype=np.float32)
    for k in range(256):
        j = k // 32
        out[k] = np.float32(d64 * sc[j] * q[k] - m64 * m[j])
    return out


def rows_of_blocks(blocks):
    """Stack a list of rows, each a list of 144-byte blocks, into a uint8 matrix."""
    return np.stack([np.frombuffer(b"".join(r), dtype=np.uint8) for r in blocks])
