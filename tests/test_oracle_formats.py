"""Pins of the oracle's other block formats (Q5_K, Q6_K, Q5_1), no GPU.

Blocks are built here from the format descriptions (GGUF arrangements; the
pages name the formats but do not lay them out), independently of the oracle:
  Q5_K, 176 bytes / 256 weights: fp16 d, fp16 dmin, 12 scale bytes packed as
    Q4_K, qh[32] (bit k/32 of qh[k%32] = bit 4 of code k), qs[128] (low
    nibbles arranged as Q4_K); w = d*sc*q - dmin*m.
  Q6_K, 210 bytes / 256 weights: ql[128], qh[64], int8 scales[16], fp16 d;
    weight k of half n (r = k%128, i = r/32, l = r%32): low 4 bits in
    ql[64n + l + 32(i&1)] (low nibble if i < 2, else high), high 2 bits at
    bits 2i..2i+1 of qh[32n + l]; w = d * scales[k/16] * (q - 32).
  Q5_1, 24 bytes / 32 weights: fp16 d, fp16 m, qh (32-bit little endian:
    bit j = bit 4 of code j), qs[16] (code j < 16 low nibble of qs[j], code
    16+j high nibble); w = d*q + m.
"""
import numpy as np
import pytest

from oracle import oracle as orc
from quantized_ffn_gb300 import synth
from tests.q4k_blocks import f16_bits, pack_codes, pack_scales

Q5K, Q6K, Q51 = orc.FMT_Q5_K, orc.FMT_Q6_K, orc.FMT_Q5_1


def u16(v):
    return bytes([v & 255, v >> 8])


def build_q5k(d, dmin, sc, m, q):
    q = [int(v) for v in q]
    assert len(q) == 256 and all(0 <= v < 32 for v in q)
    qh = [0] * 32
    for k, v in enumerate(q):
        qh[k % 32] |= (v >> 4) << (k // 32)
    blk = u16(f16_bits(d)) + u16(f16_bits(dmin)) + pack_scales(sc, m) + bytes(qh) + \
        pack_codes([v & 15 for v in q])
    assert len(blk) == 176
    return blk


def build_q6k(d, sc, q):
    q = [int(v) for v in q]
    assert len(q) == 256 and all(0 <= v < 64 for v in q) and len(sc) == 16
    ql, qh = [0] * 128, [0] * 64
    for k, v in enumerate(q):
        n, r = divmod(k, 128)
        i, l = divmod(r, 32)
        b = 64 * n + l + 32 * (i & 1)
        ql[b] |= (v & 15) << (0 if i < 2 else 4)
        qh[32 * n + l] |= (v >> 4) << (2 * i)
    blk = bytes(ql) + bytes(qh) + np.array(sc, dtype=np.int8).tobytes() + u16(f16_bits(d))
    assert len(blk) == 210
    return blk


def build_q51(d, m, q):
    q = [int(v) for v in q]
    assert len(q) == 32 and all(0 <= v < 32 for v in q)
    qh = 0
    for j, v in enumerate(q):
        qh |= (v >> 4) << j
    qs = bytes((q[j] & 15) | ((q[16 + j] & 15) << 4) for j in range(16))
    blk = u16(f16_bits(d)) + u16(f16_bits(m)) + qh.to_bytes(4, "little") + qs
    assert len(blk) == 24
    return blk


def deq(blk, fmt, cols):
    a = np.frombuffer(blk, dtype=np.uint8).reshape(1, -1)
    return orc.dequant_fmt(a, fmt, 1, cols)[0]


def test_row_bytes():
    assert orc.row_bytes_fmt(Q5K, 768) == 3 * 176 and synth.row_bytes_fmt(Q5K, 768) == 3 * 176
    assert orc.row_bytes_fmt(Q6K, 11008) == 43 * 210
    assert orc.row_bytes_fmt(Q51, 704) == 22 * 24
    assert orc.row_bytes_fmt(orc.FMT_Q4_K, 11008) == orc.row_bytes(11008)


def test_q5k_closed_form():
    sc = [j + 1 for j in range(8)]
    m = [2 * j + 1 for j in range(8)]
    q = [k % 32 for k in range(256)]
    w = deq(build_q5k(1.0, 0.5, sc, m, q), Q5K, 256)
    ref = [(k // 32 + 1) * (k % 32) - 0.5 * (2 * (k // 32) + 1) for k in range(256)]
    assert w.tolist() == ref


def test_q6k_closed_form():
    sc = [s - 8 for s in range(16)]
    q = [(7 * k) % 64 for k in range(256)]
    w = deq(build_q6k(0.25, sc, q), Q6K, 256)
    ref = [0.25 * (k // 16 - 8) * ((7 * k) % 64 - 32) for k in range(256)]
    assert w.tolist() == ref


def test_q51_closed_form_and_partial_rows():
    q = [(3 * j) % 32 for j in range(32)]
    blk = build_q51(2.0, -3.5, q)
    w = deq(blk, Q51, 32)
    assert w.tolist() == [2.0 * v - 3.5 for v in q]
    # a row of three blocks read to 80 columns: the third block's last 16 unused
    row = blk + build_q51(0.5, 1.0, q) + build_q51(4.0, 0.0, q)
    w = deq(row, Q51, 80)
    assert w[32:64].tolist() == [0.5 * v + 1.0 for v in q]
    assert w[64:80].tolist() == [4.0 * v for v in q[:16]]


@pytest.mark.parametrize("fmt", [Q5K, Q6K, Q51])
def test_high_bit_positions(fmt):
    # every weight zero but one, whose high code bit differs: exactly that
    # weight moves, by 16 steps (Q6_K: codes are stored as q + 32, so from the
    # zero code 32 bit 4 set gives +16 and bit 5 cleared gives -32)
    n = 32 if fmt == Q51 else 256
    cases = [(48, 16.0), (0, -32.0)] if fmt == Q6K else [(16, 16.0)]
    for k in range(n):
        for code, step in cases:
            if fmt == Q5K:
                q = [0] * n
                q[k] = code
                w = deq(build_q5k(1.0, 0.0, [1] * 8, [0] * 8, q), fmt, n)
            elif fmt == Q6K:
                q = [32] * n
                q[k] = code
                w = deq(build_q6k(1.0, [1] * 16, q), fmt, n)
            else:
                q = [0] * n
                q[k] = code
                w = deq(build_q51(1.0, 0.0, q), fmt, n)
            expect = np.zeros(n, np.float32)
            expect[k] = step
            assert np.array_equal(w, expect), (fmt, k, code)


def test_q6k_exact_products_exhaustive():
    # every (scale, code) with a d that uses all 11 fp16 significand bits:
    # the value is the exact product, so fp64 agrees with the fp32 result
    d = float(np.float16(1.0 + 2 ** -10 + 2 ** -3))
    for s in range(-128, 128):
        sc = [s] * 16
        q = [(k * 37 + s) % 64 for k in range(256)]
        w = deq(build_q6k(d, sc, q), Q6K, 256)
        ref = np.array([d * s * (v - 32) for v in q], dtype=np.float64)
        assert np.array_equal(w.astype(np.float64), ref)


def test_q5k_and_q51_single_rounding():
    # w = exact product, then one fp32 rounding of the sum with the offset
    rng = np.random.default_rng(3)
    for _ in range(50):
        d = float(np.float16(abs(rng.normal(0, 1e-2))))
        dmin = float(np.float16(abs(rng.normal(0, 1e-2))))
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        q = rng.integers(0, 32, 256)
        w = deq(build_q5k(d, dmin, sc, m, q), Q5K, 256)
        ref = [np.float32(d * sc[k // 32] * q[k] - dmin * m[k // 32]) for k in range(256)]
        assert np.array_equal(w, np.array(ref, np.float32))
        mm = float(np.float16(rng.normal(0, 1e-2)))
        q = rng.integers(0, 32, 32)
        w = deq(build_q51(d, mm, q), Q51, 32)
        assert np.array_equal(w, np.array([np.float32(d * v + mm) for v in q], np.float32))


@pytest.mark.parametrize("fmt", [orc.FMT_Q4_K, Q5K, Q6K, Q51])
def test_block_with_down_format_reduces_to_matmuls(fmt):
    # the block with W_down in any format = numpy fp64 matmuls on the
    # dequantised matrices (each dequantisation pinned above)
    rng = np.random.default_rng(40 + fmt)
    T, H, I = 3, 256, 320
    Wg = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wu = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wd = synth.random_blocks(rng, fmt, H, I, 1e-2)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    g = xf @ orc.q4k_dequant(Wg, I, H).astype(np.float64).T
    u = xf @ orc.q4k_dequant(Wu, I, H).astype(np.float64).T
    h = g / (1.0 + np.exp(-g)) * u
    ref = h @ orc.dequant_fmt(Wd, fmt, H, I).astype(np.float64).T
    y = orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I, wd_fmt=fmt)
    np.testing.assert_allclose(y, ref, rtol=1e-9, atol=1e-12)
    # a routed layer of one expert with weight 1 is the same block
    ids = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1), np.float32)
    ym = orc.moe_swiglu_ffn(x, ids, w, Wg[None], Wu[None], Wd[None], T, H, I, 1, 1, wd_fmt=fmt)
    np.testing.assert_allclose(ym, y, rtol=1e-12, atol=0)
