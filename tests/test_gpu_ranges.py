"""Value ranges of the 16-bit operands on the GPU, against the oracle.

The tensor-core prefill path multiplies fp16 operands: x, the unpacked
W_gate and W_up, 16 times the unpacked W_down, and the SwiGLU intermediate
divided by 16.  Its header states the ranges that stay finite: W_down
sub-blocks up to d*sc = 8 and dmin*m = 4094, intermediates up to 1.05e6.
These tests put weights and intermediates near those limits (well outside
quantised LLM weights) and check every path -- the single-token kernels, the
single-CTA tensor-core kernel and the CTA-pair kernel -- against the oracle.
"""
import numpy as np
import pytest

from oracle import oracle as orc
from quantized_ffn_gb300 import synth, zffn
from tests.gpu_util import assert_close, dev, x_dev

pytestmark = pytest.mark.gpu

H, I = 512, 768


def _set_headers(W, rows, cols, rng, d_range, dmin_range):
    """Overwrite every block's d and dmin with fp16 values drawn uniformly
    from the given ranges (scales, mins and codes stay uniform random)."""
    nb = cols // 256
    blk = W.reshape(rows, nb, 144)
    d = rng.uniform(*d_range, size=(rows, nb)).astype(np.float16)
    dm = rng.uniform(*dmin_range, size=(rows, nb)).astype(np.float16)
    blk[:, :, 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
    blk[:, :, 2:4] = dm.view(np.uint8).reshape(rows, nb, 2)
    return W


def _intermediate(x, Wg, Wu):
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    g = xf @ orc.q4k_dequant(Wg, I, H).astype(np.float64).T
    u = xf @ orc.q4k_dequant(Wu, I, H).astype(np.float64).T
    return g / (1.0 + np.exp(-np.clip(g, -700, 700))) * u


@pytest.mark.parametrize("T", [1, 40, 300])
def test_down_weights_near_the_fp16_limit(T):
    # d*sc up to 0.12*63 = 7.6 and dmin*m up to 64*63 = 4032: W_down values
    # up to about 4000 in magnitude, 16 times that just inside fp16
    rng = np.random.default_rng(500 + T)
    Wg = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wu = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wd = _set_headers(synth.random_q4k_blocks(rng, H, I, 1e-2), H, I, rng, (0.08, 0.12), (40.0, 64.0))
    assert np.abs(orc.q4k_dequant(Wd, H, I)).max() > 3000.0
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    y = zffn.swiglu_q4k(x_dev(x), dev(Wg), dev(Wu), dev(Wd), I)
    assert zffn.get_device_error() == zffn.OK
    assert_close(y, orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I), f"large W_down T={T}")


@pytest.mark.parametrize("T", [1, 40, 300])
def test_intermediate_near_the_fp16_limit(T):
    # gate/up weights and x large enough that |h| reaches 1e5 .. 1e6
    rng = np.random.default_rng(600 + T)
    Wg = synth.random_q4k_blocks(rng, I, H, 2.5e-3)
    Wu = synth.random_q4k_blocks(rng, I, H, 2.5e-3)
    Wd = synth.random_q4k_blocks(rng, H, I, 1e-2)
    x = synth.f32_to_bf16_bits(4.0 * rng.standard_normal((T, H)).astype(np.float32))
    hmax = np.abs(_intermediate(x, Wg, Wu)).max()
    assert 1e4 < hmax < 1.05e6, hmax
    y = zffn.swiglu_q4k(x_dev(x), dev(Wg), dev(Wu), dev(Wd), I)
    assert zffn.get_device_error() == zffn.OK
    assert_close(y, orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I), f"large h T={T} (max |h| {hmax:.3g})")
