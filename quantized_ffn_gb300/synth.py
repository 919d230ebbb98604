"""Seeded synthetic inputs for the feed-forward workloads.

This module only draws random numbers and rounds them to the storage types the
library consumes (bf16 activations, fp16 block scales, raw bytes); it holds
none of the block's arithmetic.  Both the CPU oracle (in the tests) and the
GPU path (tests and benchmark) take their inputs from here, so the two sides
see the same bytes.  Weights of the quantised workloads are returned as fp32;
turning them into Q4_K blocks is the caller's job (the oracle's quantiser on
the CPU side, ``zffn_q4k_quantize`` on the GPU side; the two are bit-identical).

Workloads (shapes of a Qwen3.5-9B-like layer, H=4096, I=11008, and of a
128-expert MoE layer, as on the source pages):

=========  =====================================================================
tiny       T=16, H=256, I=704; Q4_K blocks drawn directly: 4-bit codes and
           6-bit scales/mins uniform (uniform random bytes), d and dmin =
           fp16(|N(0, 1e-3)|); x = bf16(N(0, 1)); seed 0
prefill    H=4096, I=11008; W_gate, W_up [I, H], W_down [H, I] fp32 ~ N(0, 0.02)
           then x [T, H] = bf16(N(0, 1)); T=256 seed 1, T=2048 seed 2 where
           round(1% of T) distinct rows (chosen by the generator) are scaled by
           20 before rounding to bf16
decode     the same layer drawn with seed 3, then 1000 tokens x_t ~ N(0, 1)
moe        E=128 experts, H=2048, I=768, top_k=8; expert e's W_gate, W_up,
           W_down drawn from child stream e of SeedSequence(4); router logits
           [T, 128] ~ N(0, 1) and x from child stream E; the expert ids and
           weights are not drawn: the router turns the logits into them (the
           8 largest logits, softmax over those 8)
=========  =====================================================================
"""
from __future__ import annotations

import numpy as np

QK = 256
QK_BYTES = 144


def row_bytes(cols: int) -> int:
    return ((cols + QK - 1) // QK) * QK_BYTES


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the 16-bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def random_q4k_blocks(rng: np.random.Generator, rows: int, cols: int,
                      dscale: float = 1e-3) -> np.ndarray:
    """Random Q4_K rows: uniform code/scale bytes, d and dmin = fp16(|N(0, dscale)|).

    Uniform random bytes make every 4-bit code and every 6-bit scale/min
    uniform on its range whatever the bit arrangement.
    """
    nb = (cols + QK - 1) // QK
    d = np.abs(rng.normal(0.0, dscale, size=(rows, nb))).astype(np.float16)
    dmin = np.abs(rng.normal(0.0, dscale, size=(rows, nb))).astype(np.float16)
    scales = rng.integers(0, 256, size=(rows, nb, 12), dtype=np.uint8)
    qs = rng.integers(0, 256, size=(rows, nb, 128), dtype=np.uint8)
    out = np.empty((rows, nb, QK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:4] = dmin.view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 4:16] = scales
    out[:, :, 16:144] = qs
    return out.reshape(rows, nb * QK_BYTES)


# block formats of W_down on the single-token paths: code, weights and bytes
# per block
FMT_Q4_K, FMT_Q5_K, FMT_Q6_K, FMT_Q5_1 = 0, 1, 2, 3
FMT_BLOCK = {FMT_Q4_K: (256, 144), FMT_Q5_K: (256, 176), FMT_Q6_K: (256, 210), FMT_Q5_1: (32, 24)}


def row_bytes_fmt(fmt: int, cols: int) -> int:
    bw, bb = FMT_BLOCK[fmt]
    return ((cols + bw - 1) // bw) * bb


def random_blocks(rng: np.random.Generator, fmt: int, rows: int, cols: int,
                  dscale: float = 1e-3) -> np.ndarray:
    """Random rows of blocks of format fmt: uniform random bytes everywhere
    except the fp16 scale fields, which get fp16(|N(0, dscale)|) (Q5_1's
    offset m: fp16(N(0, dscale)), either sign).  Uniform bytes make every code
    and every packed scale uniform on its range."""
    if fmt == FMT_Q4_K:
        return random_q4k_blocks(rng, rows, cols, dscale)
    bw, bb = FMT_BLOCK[fmt]
    nb = (cols + bw - 1) // bw
    out = rng.integers(0, 256, size=(rows, nb, bb), dtype=np.uint8)
    d = np.abs(rng.normal(0.0, dscale, size=(rows, nb))).astype(np.float16).view(np.uint8)
    d = d.reshape(rows, nb, 2)
    if fmt == FMT_Q5_K:
        out[:, :, 0:2] = d
        out[:, :, 2:4] = np.abs(rng.normal(0.0, dscale, size=(rows, nb))).astype(
            np.float16).view(np.uint8).reshape(rows, nb, 2)
    elif fmt == FMT_Q6_K:
        out[:, :, 208:210] = d
    else:
        out[:, :, 0:2] = d
        out[:, :, 2:4] = rng.normal(0.0, dscale, size=(rows, nb)).astype(
            np.float16).view(np.uint8).reshape(rows, nb, 2)
    return out.reshape(rows, nb * bb)


def tiny(seed: int = 0):
    """The tiny block: T=16, H=256, I=704; weights already in Q4_K."""
    T, H, I = 16, 256, 704
    rng = np.random.default_rng(seed)
    Wg = random_q4k_blocks(rng, I, H)
    Wu = random_q4k_blocks(rng, I, H)
    Wd = random_q4k_blocks(rng, H, I)
    x = f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    return dict(T=T, H=H, I=I, x=x, Wg=Wg, Wu=Wu, Wd=Wd)


def dense_layer_f32(rng: np.random.Generator, H: int, I: int, std: float = 0.02):
    """fp32 W_gate [I, H], W_up [I, H], W_down [H, I] ~ N(0, std), in that order."""
    Wg = rng.standard_normal((I, H), dtype=np.float32) * np.float32(std)
    Wu = rng.standard_normal((I, H), dtype=np.float32) * np.float32(std)
    Wd = rng.standard_normal((H, I), dtype=np.float32) * np.float32(std)
    return Wg, Wu, Wd


def activations(rng: np.random.Generator, T: int, H: int, outlier_frac: float = 0.0,
                outlier_scale: float = 20.0) -> np.ndarray:
    x = rng.standard_normal((T, H), dtype=np.float32)
    n_out = int(round(outlier_frac * T))
    if n_out:
        rows = rng.choice(T, size=n_out, replace=False)
        x[rows] *= np.float32(outlier_scale)
    return f32_to_bf16_bits(x)


def prefill(T: int, seed: int, H: int = 4096, I: int = 11008, outlier_frac: float = 0.0):
    """A dense layer (fp32 weights) and bf16 activations for a prefill of T tokens."""
    rng = np.random.default_rng(seed)
    Wg, Wu, Wd = dense_layer_f32(rng, H, I)
    x = activations(rng, T, H, outlier_frac)
    return dict(T=T, H=H, I=I, x=x, Wg_f32=Wg, Wu_f32=Wu, Wd_f32=Wd)


def prefill_256():
    return prefill(256, seed=1)


def prefill_2048():
    return prefill(2048, seed=2, outlier_frac=0.01)


def decode(n_tokens: int = 1000, seed: int = 3, H: int = 4096, I: int = 11008):
    """A dense layer and n_tokens single-token activations (one row per call)."""
    rng = np.random.default_rng(seed)
    Wg, Wu, Wd = dense_layer_f32(rng, H, I)
    x = activations(rng, n_tokens, H)
    return dict(T=1, H=H, I=I, n_tokens=n_tokens, x=x, Wg_f32=Wg, Wu_f32=Wu, Wd_f32=Wd)


class MoE:
    """The 128-expert workload; expert weights are drawn lazily, one expert at a time."""

    def __init__(self, T: int, seed: int = 4, E: int = 128, H: int = 2048, I: int = 768,
                 top_k: int = 8):
        self.T, self.E, self.H, self.I, self.top_k = T, E, H, I, top_k
        self._children = np.random.SeedSequence(seed).spawn(E + 1)
        rng = np.random.default_rng(self._children[E])
        logits = rng.standard_normal((T, E), dtype=np.float32)
        self.x = activations(rng, T, H)
        self.logits = logits

    def expert_f32(self, e: int):
        rng = np.random.default_rng(self._children[e])
        return dense_layer_f32(rng, self.H, self.I)

