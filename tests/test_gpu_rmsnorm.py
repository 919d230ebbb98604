"""The normalisation before the block and the pre-norm block with its
residual connection, on the GPU through the C ABI, against the oracle.

RMSNorm: the GPU sums squares and scales in fp32, the oracle in fp64, and both
round once to bf16.  The fp32 path is within a few fp32 ulps of the exact
value, far below the bf16 step (2^-8 relative), so the two agree exactly
except where the exact value lies within those few ulps of a bf16 midpoint:
there they may differ by one bf16 step.  The test requires |difference| <= one
step everywhere and exact agreement on at least 99.9 % of the elements.

The pre-norm block: the GPU's h_out - h_in is compared with the oracle's block
output on the oracle's own normalised input, at the block's tolerance."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_ffn_gb300 import synth, zffn
from tests.gpu_util import assert_close, dense_layer, dev

pytestmark = pytest.mark.gpu

EPS = 1e-6


def residual_stream(seed, T, H, scale=1.0):
    rng = np.random.default_rng(seed)
    h = (rng.standard_normal((T, H)) * scale).astype(np.float32)
    h[::3] *= np.float32(20.0)                 # rows of different magnitude
    gamma = (1.0 + 0.2 * rng.standard_normal(H)).astype(np.float32)
    return h, gamma


def bf16_vals(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def compare_bf16(got_bits, ref_bits):
    g, r = bf16_vals(got_bits), bf16_vals(ref_bits)
    step = np.abs(r) * 2.0 ** -7 + 1e-30          # one bf16 step at |r| (upper bound)
    assert np.all(np.abs(g.astype(np.float64) - r) <= step)
    assert np.mean(got_bits == ref_bits) >= 0.999


@pytest.mark.parametrize("T,H", [(1, 4096), (7, 256), (256, 4096), (3, 16384), (33, 2048)])
def test_rmsnorm_matches_oracle(T, H):
    h, gamma = residual_stream(T * 131 + H, T, H)
    x = zffn.rmsnorm_bf16(dev(h), dev(gamma), EPS)
    torch.cuda.synchronize()
    got = x.view(torch.int16).cpu().numpy().view(np.uint16)
    compare_bf16(got, orc.rmsnorm_bf16(h, gamma, EPS))


def test_rmsnorm_special_rows():
    H = 256
    h = np.zeros((4, H), np.float32)
    h[1] = 3.0                                  # constant row -> gamma (eps = 0 below)
    h[2, ::2], h[2, 1::2] = 1e-3, -1e-3         # tiny values: eps dominates
    h[3] = np.linspace(-50, 50, H, dtype=np.float32)
    gamma = np.ones(H, np.float32)
    for eps in (0.0, 1e-6, 0.5):
        hh = h if eps > 0 else h[1:]
        x = zffn.rmsnorm_bf16(dev(hh), dev(gamma), eps)
        torch.cuda.synchronize()
        got = x.view(torch.int16).cpu().numpy().view(np.uint16)
        compare_bf16(got, orc.rmsnorm_bf16(hh, gamma, eps))
    x = zffn.rmsnorm_bf16(dev(h[1:2]), dev(gamma), 0.0)
    assert torch.all(x.float() == 1.0)


def test_prenorm_block_tiny():
    d = synth.tiny()
    h, gamma = residual_stream(5, d["T"], d["H"])
    hd = dev(h)
    zffn.swiglu_q4k_prenorm_residual(hd, dev(gamma), EPS, dev(d["Wg"]), dev(d["Wu"]), dev(d["Wd"]),
                                     d["I"])
    assert zffn.get_device_error() == zffn.OK
    out_ref, x_ref = orc.prenorm_swiglu_residual(h, gamma, EPS, d["Wg"], d["Wu"], d["Wd"], d["I"])
    delta = hd.cpu().double() - torch.from_numpy(h).double()
    assert_close(delta, out_ref - h.astype(np.float64), "pre-norm block, tiny")


@pytest.mark.parametrize("T", [1, 3])
def test_prenorm_block_full_size(T):
    # the 4096 / 11008 layer (seed 1 weights): T = 1 runs the single-token
    # kernels, T = 3 the tensor-core kernel
    L = dense_layer(1, T=256)
    h, gamma = residual_stream(40 + T, T, L["H"])
    hd = dev(h)
    zffn.swiglu_q4k_prenorm_residual(hd, dev(gamma), EPS, dev(L["Wg"]), dev(L["Wu"]), dev(L["Wd"]),
                                     L["I"])
    assert zffn.get_device_error() == zffn.OK
    out_ref, _ = orc.prenorm_swiglu_residual(h, gamma, EPS, L["Wg"], L["Wu"], L["Wd"], L["I"])
    delta = hd.cpu().double() - torch.from_numpy(h).double()
    assert_close(delta, out_ref - h.astype(np.float64), f"pre-norm block T={T}")


@pytest.mark.parametrize("H,I", [(256, 704), (1024, 1472), (2048, 5632), (8192, 2048)])
def test_prenorm_single_token_norm_in_gate_up_kernel(H, I):
    # one token: the normalisation runs inside the gate/up kernel; against the
    # oracle, and against the two public steps (same x up to the order of the
    # sum of squares: an x element may round to the neighbouring bf16 value)
    rng = np.random.default_rng(H + I)
    W = [synth.random_q4k_blocks(rng, I, H, 1e-2), synth.random_q4k_blocks(rng, I, H, 1e-2),
         synth.random_q4k_blocks(rng, H, I, 1e-2)]
    h, gamma = residual_stream(H + I, 1, H, scale=3.0)
    gamma = (gamma * np.float32(1.5)).astype(np.float32)
    hd = dev(h)
    zffn.swiglu_q4k_prenorm_residual(hd, dev(gamma), EPS, *[dev(w) for w in W], I)
    assert zffn.get_device_error() == zffn.OK
    out_ref, _ = orc.prenorm_swiglu_residual(h, gamma, EPS, *W, I)
    delta = hd.cpu().double() - torch.from_numpy(h).double()
    assert_close(delta, out_ref - h.astype(np.float64), f"pre-norm T=1 H={H} I={I}")
    b = dev(h)
    x = zffn.rmsnorm_bf16(b, dev(gamma), EPS)
    zffn.swiglu_q4k(x, *[dev(w) for w in W], I, y=b, residual=True)
    torch.cuda.synchronize()
    assert_close(hd - dev(h), (b - dev(h)).cpu().double().numpy(), "folded norm vs the two steps")


def test_prenorm_block_equals_norm_then_residual_block():
    # the composed entry equals its two public steps run by hand
    d = synth.tiny()
    h, gamma = residual_stream(6, d["T"], d["H"])
    W = [dev(d[n]) for n in ("Wg", "Wu", "Wd")]
    a = dev(h)
    zffn.swiglu_q4k_prenorm_residual(a, dev(gamma), EPS, *W, d["I"])
    b = dev(h)
    x = zffn.rmsnorm_bf16(b, dev(gamma), EPS)
    zffn.swiglu_q4k(x, *W, d["I"], y=b, residual=True)
    torch.cuda.synchronize()
    # the same kernels on the same inputs; only the order of the fp32
    # reductions into h may differ
    assert torch.allclose(a, b, rtol=1e-5, atol=1e-6)
