"""Edge sizes of the block on the GPU against the oracle: the largest hidden
and intermediate widths the entry points accept, the largest expert count and
top_k, and a token count past the headline (more work units than one pass of
the persistent schedule).  Large token counts are checked on sampled rows
(tokens are independent)."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_ffn_gb300 import synth, zffn
from tests.gpu_util import assert_close, dense_layer, dev, x_dev

pytestmark = pytest.mark.gpu


def layer(seed, H, I, dscale=1e-2):
    rng = np.random.default_rng(seed)
    return (synth.random_q4k_blocks(rng, I, H, dscale), synth.random_q4k_blocks(rng, I, H, dscale),
            synth.random_q4k_blocks(rng, H, I, dscale))


def tokens(seed, T, H):
    return synth.f32_to_bf16_bits(np.random.default_rng(seed).standard_normal((T, H)).astype(np.float32))


def check_rows(x, W, H, I, rows, what):
    Wg, Wu, Wd = W
    y = zffn.swiglu_q4k(x_dev(x), dev(Wg), dev(Wu), dev(Wd), I)
    assert zffn.get_device_error() == zffn.OK
    ref = orc.swiglu_ffn(x[rows].copy(), Wg, Wu, Wd, len(rows), H, I)
    assert_close(y[rows], ref, what)


@pytest.mark.parametrize("T", [1, 40, 300])
def test_largest_hidden_width(T):
    # H = 16384: 256 gate/up K steps and 128 down jobs per unit
    H, I = 16384, 512
    W = layer(101, H, I)
    x = tokens(102 + T, T, H)
    rows = sorted({0, T // 2, T - 1} | ({127, 128, 255, 256} if T > 256 else set()))
    check_rows(x, W, H, I, rows, f"H=16384 T={T}")


@pytest.mark.parametrize("T", [1, 3, 260])
def test_largest_intermediate_width(T):
    # I = 65536: 256 intermediate chunks, W_down rows of 36,864 bytes
    H, I = 256, 65536
    W = layer(103, H, I)
    x = tokens(104 + T, T, H)
    rows = sorted({0, T // 2, T - 1} | ({255, 256} if T > 256 else set()))
    check_rows(x, W, H, I, rows, f"I=65536 T={T}")


def test_token_count_past_the_headline():
    # T = 4096 on the 4096 / 11008 layer: 16 token tiles x 43 chunks = 688
    # work units over the CTA pairs, about nine passes of the schedule
    L = dense_layer(1, T=256)
    T = 4096
    x = tokens(105, T, L["H"])
    check_rows(x, (L["Wg"], L["Wu"], L["Wd"]), L["H"], L["I"], [0, 255, 256, 2047, 2048, 4095],
               "T=4096 sampled")


@pytest.mark.parametrize("T,matvec", [(5, 0), (1, 1)])
def test_largest_expert_count_and_top_k(T, matvec):
    # E = 4096 experts (the route kernel's counts need more than 48 KB of
    # shared memory), top_k = 64
    E, H, I, k = 4096, 256, 64, 64
    rng = np.random.default_rng(106)
    Wg = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wu = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wd = np.stack([synth.random_q4k_blocks(rng, H, I, 1e-2) for _ in range(E)])
    ids, w = orc.route_top_k(rng.standard_normal((T, E)).astype(np.float32), k)
    x = tokens(107, T, H)
    old = zffn.set_option(zffn.OPT_MATVEC_MAX_T, matvec)
    try:
        y = zffn.moe_swiglu_q4k(x_dev(x), dev(ids), dev(w), dev(Wg), dev(Wu), dev(Wd), I, E)
        assert zffn.get_device_error() == zffn.OK
    finally:
        zffn.set_option(zffn.OPT_MATVEC_MAX_T, old)
    ref = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k)
    assert_close(y, ref, f"E=4096 top_k=64 T={T}")
