"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against the format's definition, a closed form, an
invariant of the block, or a special case that reduces to a library routine,
chosen so that a dropped term, a wrong sign, a wrong index or a transposed
operand in the oracle fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

from oracle import oracle as orc
from quantized_ffn_gb300 import synth
from tests.q4k_blocks import block_values, f16_bits, make_block, pack_scales, rows_of_blocks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- scalar formats ----------------------------------------------------------

def test_f16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([orc.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f16_encode_round_to_nearest_even():
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(1e-3),
        rng.standard_normal(20000).astype(np.float32) * np.float32(100.0),
        (rng.random(5000).astype(np.float32) * np.float32(6e-5)),
        np.array([0.0, -0.0, 65504.0, 65520.0, 1e9, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                  1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11], dtype=np.float32)])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([orc.f32_to_f16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_decode():
    for f in (1.0, -2.5, 3.140625, 0.0, 1e-20):
        b = synth.f32_to_bf16_bits(np.array([f], dtype=np.float32))[0]
        assert orc.bf16_to_f32(int(b)) == float(synth.bf16_bits_to_f32(np.array([b]))[0])
    assert orc.bf16_to_f32(0x3F80) == 1.0
    assert orc.bf16_to_f32(0xC020) == -2.5


# ---- Q4_K unpack -------------------------------------------------------------

# (byte, bit) of the 12 scale bytes -> (field, sub-block, bit of the 6-bit value),
# field 0 = scale, 1 = min; written out from the packing table in q4k_blocks.py.
def _expected_scale_bit(byte, bit):
    if byte < 4:
        return (0, byte, bit) if bit < 6 else (0, byte + 4, bit - 2)
    if byte < 8:
        return (1, byte - 4, bit) if bit < 6 else (1, byte, bit - 2)
    j = byte - 4
    return (0, j, bit) if bit < 4 else (1, j, bit - 4)


def test_scale_min_every_bit_position():
    for byte in range(12):
        for bit in range(8):
            s = bytearray(12)
            s[byte] = 1 << bit
            field, sub, vbit = _expected_scale_bit(byte, bit)
            for j in range(8):
                sc, m = orc.scale_min(bytes(s), j)
                want_sc = (1 << vbit) if (field == 0 and j == sub) else 0
                want_m = (1 << vbit) if (field == 1 and j == sub) else 0
                assert (sc, m) == (want_sc, want_m), (byte, bit, j)


def test_scale_min_roundtrip_all_values():
    rng = np.random.default_rng(5)
    for _ in range(200):
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        packed = pack_scales(sc, m)
        for j in range(8):
            assert orc.scale_min(packed, j) == (sc[j], m[j])


def test_code_nibble_positions():
    # one non-zero code at each position k, d=1, dmin=0, all scales 1
    for k in range(256):
        q = [0] * 256
        q[k] = 7
        blk = make_block(1.0, 0.0, [1] * 8, [0] * 8, q)
        out = orc.q4k_dequant(np.frombuffer(blk, dtype=np.uint8), 1, 256)[0]
        nz = np.nonzero(out)[0]
        assert list(nz) == [k] and out[k] == 7.0


def test_hand_built_block_closed_form():
    # d = 1, dmin = 0.5, sc_j = j+1, m_j = 2j, q_k = k mod 16:
    # w_k = (j+1) * (k mod 16) - j   with j = k // 32
    q = [k % 16 for k in range(256)]
    blk = make_block(1.0, 0.5, [j + 1 for j in range(8)], [2 * j for j in range(8)], q)
    out = orc.q4k_dequant(np.frombuffer(blk, dtype=np.uint8), 1, 256)[0]
    want = np.array([(k // 32 + 1) * (k % 16) - (k // 32) for k in range(256)], dtype=np.float32)
    assert np.array_equal(out, want)


def test_min_is_subtracted():
    # all codes 0: w = -dmin * m
    blk = make_block(0.25, 0.125, [3] * 8, list(range(8)), [0] * 256)
    out = orc.q4k_dequant(np.frombuffer(blk, dtype=np.uint8), 1, 256)[0]
    assert np.array_equal(out, np.repeat(-0.125 * np.arange(8), 32).astype(np.float32))


@pytest.mark.parametrize("d,dmin", [(1.0, 1.0), (0.000123, 0.00456), (2.0 ** -24, 3 * 2.0 ** -24),
                                    (65504.0, 0.5), (0.3, 0.0)])
def test_exhaustive_code_scale_min(d, dmin):
    # every (q, sc, m): 64*64 (sc, m) pairs, one sub-block each, codes 0..15 twice
    blocks, want = [], []
    pairs = [(s, m) for s in range(64) for m in range(64)]
    q = [(k % 32) % 16 for k in range(256)]
    for i in range(0, len(pairs), 8):
        sc = [p[0] for p in pairs[i:i + 8]]
        mm = [p[1] for p in pairs[i:i + 8]]
        blocks.append(make_block(d, dmin, sc, mm, q))
        want.append(block_values(d, dmin, sc, mm, q))
    buf = np.frombuffer(b"".join(blocks), dtype=np.uint8)
    out = orc.q4k_dequant(buf, len(blocks), 256)
    want = np.stack(want)
    assert np.array_equal(out.view(np.uint32), want.view(np.uint32))


def test_partial_last_block():
    rng = np.random.default_rng(1)
    rows = synth.random_q4k_blocks(rng, 3, 704)
    full = orc.q4k_dequant(rows, 3, 768)
    part = orc.q4k_dequant(rows, 3, 704)
    assert np.array_equal(part, full[:, :704])


# ---- quantiser ---------------------------------------------------------------

def _split_blocks(b):
    b = b.reshape(-1, 144)
    d = b[:, 0:2].copy().view(np.float16).astype(np.float32)[:, 0]
    dmin = b[:, 2:4].copy().view(np.float16).astype(np.float32)[:, 0]
    sc = np.zeros((len(b), 8), dtype=np.int64)
    m = np.zeros((len(b), 8), dtype=np.int64)
    for i in range(len(b)):
        for j in range(8):
            sc[i, j], m[i, j] = orc.scale_min(bytes(b[i, 4:16]), j)
    return d, dmin, sc, m


def test_quantizer_roundtrip_bound():
    rng = np.random.default_rng(2)
    w = rng.standard_normal((16, 512)).astype(np.float32) * np.float32(0.02)
    w[3] += np.float32(0.05)          # all-positive-ish row
    w[4] -= np.float32(0.05)          # all-negative-ish row
    b = orc.q4k_quantize(w)
    wh = orc.q4k_dequant(b, 16, 512)
    d, dmin, sc, m = _split_blocks(b)
    err = np.abs(wh - w).reshape(-1, 8, 32)
    ds = (d[:, None] * sc).astype(np.float64)
    # |w - w_hat| <= d*sc/2 (code rounding) + 15*d/2 (scale rounding, clamped top code)
    #               + dmin/2 (min rounding), plus fp32 rounding slack
    bound = ds / 2 + 7.5 * d[:, None] + dmin[:, None] / 2 + 1e-6
    assert np.all(err <= bound[:, :, None])


def test_quantizer_rounds_to_nearest_code():
    # rint, not floor: the RMS code-rounding error of Gaussian data is about
    # step/sqrt(12) ~ 0.29 step (floor would give ~0.58 and a bias)
    rng = np.random.default_rng(3)
    w = rng.standard_normal((64, 1024)).astype(np.float32) * np.float32(0.02)
    b = orc.q4k_quantize(w)
    wh = orc.q4k_dequant(b, 64, 1024)
    d, dmin, sc, m = _split_blocks(b)
    step = np.repeat((d[:, None] * sc).reshape(-1), 32).reshape(w.shape)
    r = (wh - w) / step
    assert 0.22 < np.sqrt(np.mean(r ** 2)) < 0.36
    assert abs(np.mean(r)) < 0.05


def test_quantizer_zero_and_constant_blocks():
    z = orc.q4k_quantize(np.zeros((1, 256), dtype=np.float32))
    assert not z.any()
    c = np.full((1, 256), 0.75, dtype=np.float32)
    bc = orc.q4k_quantize(c)
    d, dmin, sc, m = _split_blocks(bc)
    assert dmin[0] == 0 and np.all(m == 0) and np.all(sc == 63)
    wh = orc.q4k_dequant(bc, 1, 256)
    assert np.all(np.abs(wh - 0.75) <= 7.5 * d[0] + 1e-6)


def test_quantizer_tail_is_zero_padded():
    rng = np.random.default_rng(4)
    w = rng.standard_normal((2, 300)).astype(np.float32)
    padded = np.zeros((2, 512), dtype=np.float32)
    padded[:, :300] = w
    assert np.array_equal(orc.q4k_quantize(w), orc.q4k_quantize(padded))


# ---- silu --------------------------------------------------------------------

def test_silu_closed_forms():
    assert orc.silu(0.0) == 0.0
    # textbook logistic values: sigma(2) = 0.88079707797788244..., sigma(-2) = 0.11920292202211756...
    assert math.isclose(orc.silu(2.0), 2 * 0.8807970779778824, rel_tol=1e-15)
    assert math.isclose(orc.silu(-2.0), -2 * 0.11920292202211755, rel_tol=1e-15)
    assert math.isclose(orc.silu(50.0), 50.0, rel_tol=1e-15)
    assert abs(orc.silu(-50.0)) < 1e-19


# ---- the feed-forward block ----------------------------------------------------

def _rand_rows(seed, rows, cols, dscale=1e-2):
    return synth.random_q4k_blocks(np.random.default_rng(seed), rows, cols, dscale)


def _x(seed, T, H):
    return synth.f32_to_bf16_bits(np.random.default_rng(seed).standard_normal((T, H)).astype(np.float32))


def test_zero_input_gives_zero_output():
    H, I = 256, 512
    Wg, Wu, Wd = _rand_rows(1, I, H), _rand_rows(2, I, H), _rand_rows(3, H, I)
    y = orc.swiglu_ffn(np.zeros((3, H), np.uint16), Wg, Wu, Wd, 3, H, I)
    assert np.all(y == 0.0)


@pytest.mark.parametrize("which", ["gate", "up", "down"])
def test_zero_weights_give_zero_output(which):
    H, I, T = 256, 512, 4
    W = {"gate": _rand_rows(1, I, H), "up": _rand_rows(2, I, H), "down": _rand_rows(3, H, I)}
    W[which] = np.zeros_like(W[which])           # d = dmin = 0
    y = orc.swiglu_ffn(_x(9, T, H), W["gate"], W["up"], W["down"], T, H, I)
    assert np.all(y == 0.0)


def test_one_hot_input_selects_weight_columns():
    H, I, T = 512, 256, 3
    Wg, Wu, Wd = _rand_rows(1, I, H), _rand_rows(2, I, H), _rand_rows(3, H, I)
    cols = [0, 300, 511]
    x = np.zeros((T, H), dtype=np.uint16)
    for t, c in enumerate(cols):
        x[t, c] = 0x3F80                          # bf16 1.0
    y = orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I)
    g = orc.q4k_dequant(Wg, I, H)
    u = orc.q4k_dequant(Wu, I, H)
    dn = orc.q4k_dequant(Wd, H, I).astype(np.float64)
    for t, c in enumerate(cols):
        gc = g[:, c].astype(np.float64)
        h = gc / (1 + np.exp(-gc)) * u[:, c]
        np.testing.assert_allclose(y[t], dn @ h, rtol=1e-12, atol=1e-300)


def test_large_gate_reduces_to_bilinear_matmul():
    # with every gate pre-activation >= 40, silu(g) = g to fp64 precision, so the
    # block is y = Wd ((Wg x) * (Wu x)): a chain of plain matrix products.
    H, I, T = 512, 320, 5
    rng = np.random.default_rng(7)
    rows = []
    for i in range(I):
        blks = []
        for b in range(H // 256):
            q = rng.integers(1, 16, 256)
            blks.append(make_block(0.25, 0.0, rng.integers(1, 64, 8), [0] * 8, q))
        rows.append(blks)
    Wg = rows_of_blocks(rows)
    Wu, Wd = _rand_rows(8, I, H), _rand_rows(9, H, I)
    xf = (1.0 + 0.5 * rng.integers(0, 2, (T, H))).astype(np.float32)   # 1.0 or 1.5
    x = synth.f32_to_bf16_bits(xf)
    y = orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I)
    G = orc.q4k_dequant(Wg, I, H).astype(np.float64)
    U = orc.q4k_dequant(Wu, I, H).astype(np.float64)
    D = orc.q4k_dequant(Wd, H, I).astype(np.float64)
    X = xf.astype(np.float64)
    g = X @ G.T
    assert g.min() >= 40.0
    want = ((g * (X @ U.T)) @ D.T)
    np.testing.assert_allclose(y, want, rtol=1e-11, atol=1e-12 * np.abs(want).max())


def test_tokens_are_independent():
    H, I, T = 256, 704, 6
    Wg, Wu, Wd = _rand_rows(1, I, H), _rand_rows(2, I, H), _rand_rows(3, H, I)
    x = _x(4, T, H)
    y = orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I)
    y2 = orc.swiglu_ffn(x[2:5].copy(), Wg, Wu, Wd, 3, H, I)
    assert np.array_equal(y[2:5], y2)


def _scale_d(blocks, factor):
    # multiply d and dmin of every block by an exact power of two
    b = blocks.reshape(-1, 144).copy()
    for lo in (0, 2):
        v = b[:, lo:lo + 2].copy().view(np.float16).astype(np.float32) * np.float32(factor)
        b[:, lo:lo + 2] = v.astype(np.float16).view(np.uint8)
    return b.reshape(blocks.shape)


def test_up_and_down_are_linear():
    H, I, T = 256, 512, 3
    Wg, Wu, Wd = _rand_rows(1, I, H), _rand_rows(2, I, H), _rand_rows(3, H, I)
    x = _x(5, T, H)
    y = orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I)
    assert np.array_equal(orc.swiglu_ffn(x, Wg, _scale_d(Wu, 2.0), Wd, T, H, I), 2 * y)
    assert np.array_equal(orc.swiglu_ffn(x, Wg, Wu, _scale_d(Wd, 4.0), T, H, I), 4 * y)


def test_intermediate_block_permutation_invariance():
    # permuting the intermediate dimension in whole 256-blocks (rows of Wg/Wu and
    # the matching blocks of every Wd row) leaves y unchanged
    H, I, T = 256, 768, 4
    Wg, Wu, Wd = _rand_rows(1, I, H), _rand_rows(2, I, H), _rand_rows(3, H, I)
    x = _x(6, T, H)
    y = orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I)
    perm = [2, 0, 1]
    rp = np.concatenate([np.arange(256 * p, 256 * p + 256) for p in perm])
    Wd_b = Wd.reshape(H, 3, 144)[:, perm, :].reshape(H, 3 * 144)
    yp = orc.swiglu_ffn(x, Wg[rp].copy(), Wu[rp].copy(), np.ascontiguousarray(Wd_b), T, H, I)
    np.testing.assert_allclose(yp, y, rtol=1e-12, atol=1e-14 * np.abs(y).max())


# ---- mixture of experts ----------------------------------------------------------

def _experts(E, H, I, seed=20):
    Wg = np.stack([_rand_rows(seed + 3 * e, I, H) for e in range(E)])
    Wu = np.stack([_rand_rows(seed + 3 * e + 1, I, H) for e in range(E)])
    Wd = np.stack([_rand_rows(seed + 3 * e + 2, H, I) for e in range(E)])
    return Wg, Wu, Wd


def test_moe_single_expert_equals_dense():
    E, H, I, T = 4, 256, 320, 3
    Wg, Wu, Wd = _experts(E, H, I)
    x = _x(1, T, H)
    ids = np.array([[2], [0], [3]], dtype=np.int32)
    w = np.ones((T, 1), dtype=np.float32)
    y = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, 1)
    for t in range(T):
        e = ids[t, 0]
        yd = orc.swiglu_ffn(x[t:t + 1].copy(), Wg[e], Wu[e], Wd[e], 1, H, I)
        assert np.array_equal(y[t], yd[0])


def test_moe_identical_experts_with_unit_weight_sum_equals_dense():
    E, H, I, T, k = 5, 256, 256, 2, 3
    one = _experts(1, H, I)
    Wg, Wu, Wd = (np.repeat(a, E, axis=0) for a in one)
    x = _x(2, T, H)
    ids = np.array([[0, 3, 4], [1, 2, 0]], dtype=np.int32)
    w = np.array([[0.5, 0.25, 0.25], [0.125, 0.375, 0.5]], dtype=np.float32)
    y = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k)
    yd = orc.swiglu_ffn(x, one[0][0], one[1][0], one[2][0], T, H, I)
    np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-14 * np.abs(yd).max())


def test_moe_slot_order_and_invalid_ids():
    E, H, I, T, k = 6, 256, 256, 2, 4
    Wg, Wu, Wd = _experts(E, H, I)
    x = _x(3, T, H)
    ids = np.array([[5, 1, 2, 0], [3, 4, 1, 2]], dtype=np.int32)
    w = np.array([[0.4, 0.3, 0.2, 0.1], [0.25, 0.25, 0.3, 0.2]], dtype=np.float32)
    y = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k)
    perm = [2, 0, 3, 1]
    yp = orc.moe_swiglu_ffn(x, ids[:, perm].copy(), w[:, perm].copy(), Wg, Wu, Wd, T, H, I, E, k)
    np.testing.assert_allclose(yp, y, rtol=1e-12, atol=1e-14 * np.abs(y).max())
    bad = ids.copy()
    bad[0, 1] = -1
    bad[1, 3] = E
    yb = orc.moe_swiglu_ffn(x, bad, w, Wg, Wu, Wd, T, H, I, E, k)
    keep = orc.moe_swiglu_ffn(x, ids[:, [0, 2, 3]].copy(), w[:, [0, 2, 3]].copy(),
                              Wg, Wu, Wd, T, H, I, E, 3)
    np.testing.assert_allclose(yb[0], keep[0], rtol=1e-12, atol=1e-14 * np.abs(y).max())
    keep1 = orc.moe_swiglu_ffn(x, ids[:, [0, 1, 2]].copy(), w[:, [0, 1, 2]].copy(),
                               Wg, Wu, Wd, T, H, I, E, 3)
    np.testing.assert_allclose(yb[1], keep1[1], rtol=1e-12, atol=1e-14 * np.abs(y).max())


def test_moe_down_scale_closed_forms():
    # Per-expert scale on the down projection ("Four bottlenecks, one CUDA
    # backend...", section "Bottleneck 2"): y_t = sum_j w_tj s_e FFN_e(x_t).
    E, H, I, T, k = 5, 256, 320, 3, 3
    Wg, Wu, Wd = _experts(E, H, I, seed=40)
    x = _x(4, T, H)
    ids = np.array([[4, 1, 2], [0, 3, 1], [2, 2, 4]], dtype=np.int32)
    w = np.array([[0.5, 0.3, 0.2], [0.6, 0.25, 0.15], [0.7, 0.2, 0.1]], dtype=np.float32)
    y = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k)
    # no scale and unit scales agree exactly
    assert np.array_equal(orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k,
                                             down_scale=np.ones(E, np.float32)), y)
    # a common power-of-two scale scales the output exactly
    for p2 in (0.25, 8.0):
        ys = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k,
                                down_scale=np.full(E, p2, np.float32))
        assert np.array_equal(ys, y * p2)
    # zero scales silence the output; a zero scale on one expert equals dropping its slots
    assert not np.any(orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k,
                                         down_scale=np.zeros(E, np.float32)))
    s = np.ones(E, np.float32)
    s[2] = 0.0
    w0 = w.copy()
    w0[ids == 2] = 0.0
    np.testing.assert_array_equal(
        orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k, down_scale=s),
        orc.moe_swiglu_ffn(x, ids, w0, Wg, Wu, Wd, T, H, I, E, k))


def test_moe_down_scale_recomposed_from_dense_blocks():
    # General scales against the dense block of each chosen expert, weighted
    # by w * s in fp64 here (the dense block is pinned on its own).
    E, H, I, T, k = 4, 256, 256, 2, 2
    Wg, Wu, Wd = _experts(E, H, I, seed=50)
    x = _x(5, T, H)
    ids = np.array([[3, 0], [1, 3]], dtype=np.int32)
    w = np.array([[0.625, 0.375], [0.9, 0.1]], dtype=np.float32)
    s = np.array([1.7, -0.4, 3.0, 0.37], dtype=np.float32)
    y = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k, down_scale=s)
    for t in range(T):
        ref = np.zeros(H)
        for j in range(k):
            e = ids[t, j]
            ref += (float(w[t, j]) * float(s[e])) * orc.swiglu_ffn(
                x[t:t + 1].copy(), Wg[e], Wu[e], Wd[e], 1, H, I)[0]
        np.testing.assert_allclose(y[t], ref, rtol=1e-12, atol=1e-14 * np.abs(ref).max())


# ---- the pages' byte model ---------------------------------------------------------

def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split("=")
                vals[k.strip()] = float(v)
    return vals


def test_intermediate_byte_model_matches_pages():
    g = _golden("byte_model.txt")
    H, I = int(g["hidden"]), int(g["intermediate"])
    per_token = I * 2 / 1024                       # fp16 intermediate row, KB
    assert round(per_token, 1) == g["kb_per_token_fp16"]
    assert round(g["crossings_staged"] * per_token) == g["kb_per_token_staged"]
    # the page counts KB in units of 1024 bytes but this MB in units of 10^6 bytes
    assert round(256 * I * 2 / 1e6, 1) == g["mb_256_token_tile"]
    assert round(I / H, 1) == g["width_ratio"]
    # 4.5 bits per weight for Q4_K (144 bytes per 256 weights)
    assert 144 * 8 / 256 == g["q4k_bits_per_weight"]
    # staged dequant moves 4.5 + 16 + 16 bits per weight, the fused path 4.5
    staged = g["q4k_bits_per_weight"] + 16 + 16
    assert round(staged / g["q4k_bits_per_weight"]) == g["weight_traffic_cut"]


# ---- router: top-k ids and softmax weights ------------------------------------

def _softmax64(v):
    v = np.asarray(v, dtype=np.float64)
    e = np.exp(v - v.max())
    return e / e.sum()


def test_router_matches_stable_sort_and_softmax():
    # Integer-valued logits in a small range make ties common; a stable sort of
    # the negated logits orders equal logits by index, which is the stated
    # tie rule, so it must pick the same ids in the same order.
    rng = np.random.default_rng(21)
    for T, E, k in [(64, 128, 8), (16, 37, 5), (8, 4096, 64), (5, 3, 3)]:
        logits = rng.integers(-6, 7, size=(T, E)).astype(np.float32)
        logits[: T // 2] += rng.standard_normal((T // 2, E)).astype(np.float32)
        ids, w = orc.route_top_k(logits, k)
        order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
        assert np.array_equal(ids, order.astype(np.int32))
        for t in range(T):
            ref = _softmax64(logits[t, order[t]]).astype(np.float32)
            np.testing.assert_allclose(w[t], ref, rtol=2e-7, atol=0)


def test_router_closed_forms():
    # equal logits: the first k indices, weight 1/k each
    ids, w = orc.route_top_k(np.full((3, 10), 0.75, np.float32), 4)
    assert np.array_equal(ids, np.tile(np.arange(4, dtype=np.int32), (3, 1)))
    assert np.all(w == np.float32(0.25))
    # a single choice carries weight exactly 1
    rng = np.random.default_rng(22)
    lg = rng.standard_normal((7, 33)).astype(np.float32)
    ids, w = orc.route_top_k(lg, 1)
    assert np.array_equal(ids[:, 0], np.argmax(lg, axis=1).astype(np.int32))
    assert np.all(w == 1.0)
    # two chosen logits a > b: weights 1/(1+e^(b-a)) and e^(b-a)/(1+e^(b-a))
    lg = np.array([[0.0, 2.0, -1.0, 0.5]], np.float32)
    ids, w = orc.route_top_k(lg, 2)
    assert ids.tolist() == [[1, 3]]
    r = math.exp(0.5 - 2.0)
    np.testing.assert_allclose(w[0], [1 / (1 + r), r / (1 + r)], rtol=1e-7)
    # shifting every logit by an exact constant changes nothing
    lg = rng.integers(-20, 20, size=(4, 64)).astype(np.float32)
    a = orc.route_top_k(lg, 6)
    b = orc.route_top_k(lg + np.float32(1024.0), 6)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # the weights of a token sum to 1 within fp32 rounding
    lg = rng.standard_normal((50, 128)).astype(np.float32) * np.float32(3.0)
    _, w = orc.route_top_k(lg, 8)
    np.testing.assert_allclose(w.astype(np.float64).sum(axis=1), 1.0, rtol=0, atol=8 * 2.0 ** -24)


def test_router_special_values():
    nan, inf = np.float32("nan"), np.float32("inf")
    lg = np.array([[nan, -inf, 1.0, -0.0, 0.0, nan, -3.0]], np.float32)
    ids, w = orc.route_top_k(lg, 7)
    # numbers first (descending; -0 equals +0, so index decides), then -inf,
    # then the NaNs by index
    assert ids.tolist() == [[2, 3, 4, 6, 1, 0, 5]]
    assert np.isnan(w[0, 5]) and np.isnan(w[0, 6])
    ids, w = orc.route_top_k(lg, 4)
    assert ids.tolist() == [[2, 3, 4, 6]]
    ref = _softmax64([1.0, 0.0, 0.0, -3.0]).astype(np.float32)
    np.testing.assert_allclose(w[0], ref, rtol=2e-7)


def test_router_brute_force_over_all_orders():
    # every arrangement of a small multiset of logits (ties included): the
    # chosen ids are the k best positions under (value desc, index asc)
    import itertools
    vals = [2.0, 2.0, -1.0, 0.5, 0.5]
    for perm in set(itertools.permutations(vals)):
        lg = np.array([perm], np.float32)
        ranked = sorted(range(len(perm)), key=lambda i: (-perm[i], i))
        for k in (1, 3, 5):
            ids, _ = orc.route_top_k(lg, k)
            assert ids[0].tolist() == ranked[:k]


# ---- RMSNorm before the block, residual around it ------------------------------

def _bf16(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def test_bf16_rounding_against_float32_bits():
    # For values exact in fp32, rounding fp64 -> bf16 once equals the bit-level
    # round-to-nearest-even of the fp32 pattern (add 0x7FFF + lsb, cut).
    rng = np.random.default_rng(31)
    v = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        (rng.standard_normal(5000) * 1e4).astype(np.float32),
                        np.array([1.0, -1.0, 1 + 2 ** -8, 1 + 2 ** -9, 1 + 3 * 2 ** -9,
                                  1 + 2 ** -9 + 2 ** -20, 255.5, 0.0, -0.0], np.float32)])
    u = v.view(np.uint32)
    ref = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    got = np.array([orc.bf16_from_f64(float(a)) for a in v], dtype=np.uint16)
    assert np.array_equal(got, ref)
    # a value between two bf16 numbers that fp32 cannot hold: rounded once
    # (bf16 steps by 2^-7 on [1, 2): 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7)
    assert orc.bf16_from_f64(1 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert orc.bf16_from_f64(1 + 2 ** -8 - 2 ** -40) == 0x3F80
    assert orc.bf16_from_f64(1 + 2 ** -8) == 0x3F80 and orc.bf16_from_f64(1 + 3 * 2 ** -8) == 0x3F82


def test_rmsnorm_worked_example():
    # h = (3, 4): mean square 12.5, so x = (3, 4) / sqrt(12.5) = (0.8485, 1.1314)
    # before rounding; bf16 keeps 8 significant bits: 217/256 and 145/128.
    x = orc.rmsnorm_bf16(np.array([[3.0, 4.0]], np.float32), np.ones(2, np.float32), 0.0)
    assert _bf16(x[0]).tolist() == [217 / 256, 145 / 128]
    x = orc.rmsnorm_bf16(np.array([[3.0, 4.0]], np.float32), np.array([2.0, -0.5], np.float32), 0.0)
    assert _bf16(x[0]).tolist() == [217 / 128, -145 / 256]
    # eps enters under the root: h = (1, 1, 1, 1), eps = 3 -> 1 / sqrt(4) = 0.5
    x = orc.rmsnorm_bf16(np.ones((1, 4), np.float32), np.ones(4, np.float32), 3.0)
    assert np.all(_bf16(x[0]) == 0.5)


def test_rmsnorm_invariants():
    rng = np.random.default_rng(32)
    h = rng.standard_normal((6, 256)).astype(np.float32)
    g = np.ones(256, np.float32)
    # constant rows map to +-gamma exactly (eps = 0)
    c = np.array([[2.5] * 8, [-7.0] * 8], np.float32)
    x = orc.rmsnorm_bf16(c, np.ones(8, np.float32), 0.0)
    assert np.all(_bf16(x[0]) == 1.0) and np.all(_bf16(x[1]) == -1.0)
    # scaling a row by a power of two changes nothing (eps = 0)
    a = orc.rmsnorm_bf16(h, g, 0.0)
    b = orc.rmsnorm_bf16(h * np.float32(64.0), g, 0.0)
    assert np.array_equal(a, b)
    # gamma scales column by column: gamma = 2 doubles every value exactly
    b = orc.rmsnorm_bf16(h, np.full(256, 2.0, np.float32), 0.0)
    assert np.array_equal(_bf16(b), 2 * _bf16(a))
    # unit mean square before rounding: after it, within the bf16 step
    ms = (_bf16(a).astype(np.float64) ** 2).mean(axis=1)
    assert np.all(np.abs(ms - 1.0) < 2 ** -7)
    # a zero row stays zero when eps > 0
    x = orc.rmsnorm_bf16(np.zeros((1, 16), np.float32), np.ones(16, np.float32), 1e-6)
    assert np.all(_bf16(x) == 0.0)
    # rows are independent
    one = orc.rmsnorm_bf16(h[3:4], g, 1e-6)
    assert np.array_equal(one[0], orc.rmsnorm_bf16(h, g, 1e-6)[3])


def test_prenorm_sublayer_reduces_to_parts():
    # with zero down weights the sublayer leaves h unchanged; otherwise it is
    # h plus the block applied to the normalised rows
    d = synth.tiny()
    rng = np.random.default_rng(33)
    h = rng.standard_normal((4, d["H"])).astype(np.float32)
    gamma = (1.0 + 0.1 * rng.standard_normal(d["H"])).astype(np.float32)
    zero_wd = np.zeros_like(d["Wd"])
    out, x = orc.prenorm_swiglu_residual(h, gamma, 1e-6, d["Wg"], d["Wu"], zero_wd, d["I"])
    assert np.array_equal(out, h.astype(np.float64))
    out, x = orc.prenorm_swiglu_residual(h, gamma, 1e-6, d["Wg"], d["Wu"], d["Wd"], d["I"])
    assert np.array_equal(x, orc.rmsnorm_bf16(h, gamma, 1e-6))
    y = orc.swiglu_ffn(x, d["Wg"], d["Wu"], d["Wd"], 4, d["H"], d["I"])
    assert np.array_equal(out, h.astype(np.float64) + y)


def test_parallel_build_of_the_oracle_gives_the_same_bits():
    # The CPU baseline's all-cores leg runs the oracle's source built with
    # OpenMP: its row loops are independent and keep every sum's order, so
    # its outputs equal the single-threaded build's bit for bit.
    path = orc.build_omp()
    if path is None:
        pytest.skip("no OpenMP in this compiler")
    H, I, T = 512, 320, 3
    Wg, Wu, Wd = _rand_rows(70, I, H), _rand_rows(71, I, H), _rand_rows(72, H, I)
    x = _x(73, T, H)
    y1 = orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I)
    d1 = orc.q4k_dequant(Wg, I, H)
    prev = orc.use_library(path)
    try:
        y2 = orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I)
        d2 = orc.q4k_dequant(Wg, I, H)
    finally:
        orc.use_library(prev)
    assert np.array_equal(y1, y2) and np.array_equal(d1, d2)
