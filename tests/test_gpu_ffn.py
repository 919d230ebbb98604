"""Dense SwiGLU block on the GPU against the oracle (element by element)."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_ffn_gb300 import synth, zffn
from tests.gpu_util import assert_close, dense_layer, dev, x_dev

pytestmark = pytest.mark.gpu


def run(x_bits, Wg, Wu, Wd, I, matvec_max_t=None):
    old = None
    if matvec_max_t is not None:
        old = zffn.set_option(zffn.OPT_MATVEC_MAX_T, matvec_max_t)
    try:
        y = zffn.swiglu_q4k(x_dev(x_bits), dev(Wg), dev(Wu), dev(Wd), I)
        assert zffn.get_device_error() == zffn.OK
    finally:
        if old is not None:
            zffn.set_option(zffn.OPT_MATVEC_MAX_T, old)
    return y


def random_layer(seed, T, H, I, dscale=1e-2):
    rng = np.random.default_rng(seed)
    Wg = synth.random_q4k_blocks(rng, I, H, dscale)
    Wu = synth.random_q4k_blocks(rng, I, H, dscale)
    Wd = synth.random_q4k_blocks(rng, H, I, dscale)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    return x, Wg, Wu, Wd


def test_tiny_config_tensor_core_path():
    t = synth.tiny()
    y = run(t["x"], t["Wg"], t["Wu"], t["Wd"], t["I"], matvec_max_t=0)
    ref = orc.swiglu_ffn(t["x"], t["Wg"], t["Wu"], t["Wd"], t["T"], t["H"], t["I"])
    assert_close(y, ref, "tiny/tc")


def test_tiny_config_single_token_path():
    t = synth.tiny()
    for r in (0, 5, 15):
        x = t["x"][r:r + 1].copy()
        y = run(x, t["Wg"], t["Wu"], t["Wd"], t["I"], matvec_max_t=1)
        ref = orc.swiglu_ffn(x, t["Wg"], t["Wu"], t["Wd"], 1, t["H"], t["I"])
        assert_close(y, ref, f"tiny/matvec row {r}")


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128, 129, 255, 257, 300])
def test_tile_boundaries_tokens(T):
    H, I = 512, 704
    x, Wg, Wu, Wd = random_layer(T, T, H, I)
    y = run(x, Wg, Wu, Wd, I, matvec_max_t=0)
    assert_close(y, orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I), f"T={T}")


@pytest.mark.parametrize("H,I", [(256, 64), (256, 256), (768, 320), (1024, 1472), (2048, 768),
                                 (4096, 512)])
def test_tile_boundaries_widths(H, I):
    T = 130
    x, Wg, Wu, Wd = random_layer(H + I, T, H, I)
    y = run(x, Wg, Wu, Wd, I, matvec_max_t=0)
    assert_close(y, orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I), f"H={H} I={I}")


@pytest.mark.parametrize("H,I", [(256, 704), (1024, 1472), (2048, 768)])
def test_single_token_widths(H, I):
    x, Wg, Wu, Wd = random_layer(H * 3 + I, 1, H, I)
    y = run(x, Wg, Wu, Wd, I, matvec_max_t=1)
    assert_close(y, orc.swiglu_ffn(x, Wg, Wu, Wd, 1, H, I), f"matvec H={H} I={I}")


def test_zero_input_and_zero_weights_give_zero():
    H, I, T = 512, 704, 130
    x, Wg, Wu, Wd = random_layer(1, T, H, I)
    for path in (0, 1):
        xz = np.zeros_like(x[: (1 if path else T)])
        y = run(xz, Wg, Wu, Wd, I, matvec_max_t=path)
        assert torch.count_nonzero(y).item() == 0
        y = run(x[: (1 if path else T)].copy(), np.zeros_like(Wg), Wu, Wd, I, matvec_max_t=path)
        assert torch.count_nonzero(y).item() == 0


def test_single_token_and_prefill_paths_agree_with_oracle_on_same_rows():
    H, I = 1024, 1472
    x, Wg, Wu, Wd = random_layer(77, 4, H, I)
    ref = orc.swiglu_ffn(x, Wg, Wu, Wd, 4, H, I)
    y_tc = run(x, Wg, Wu, Wd, I, matvec_max_t=0)
    assert_close(y_tc, ref, "tc")
    for r in range(4):
        y_mv = run(x[r:r + 1].copy(), Wg, Wu, Wd, I, matvec_max_t=1)
        assert_close(y_mv, ref[r:r + 1], f"matvec row {r}")


def test_repeated_calls_are_stable():
    H, I, T = 512, 704, 200
    x, Wg, Wu, Wd = random_layer(5, T, H, I)
    ref = orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I)
    for _ in range(3):
        assert_close(run(x, Wg, Wu, Wd, I, matvec_max_t=0), ref, "repeat")


# ---- the full-size layer (H=4096, I=11008) -----------------------------------

def _sampled(layer, T, rows, matvec_max_t=0):
    Wg, Wu, Wd = dev(layer["Wg"]), dev(layer["Wu"]), dev(layer["Wd"])
    x = layer["x"][:T]
    old = zffn.set_option(zffn.OPT_MATVEC_MAX_T, matvec_max_t)
    try:
        y = zffn.swiglu_q4k(x_dev(x), Wg, Wu, Wd, layer["I"])
        assert zffn.get_device_error() == zffn.OK
    finally:
        zffn.set_option(zffn.OPT_MATVEC_MAX_T, old)
    xs = x[rows].copy()
    ref = orc.swiglu_ffn(xs, layer["Wg"], layer["Wu"], layer["Wd"], len(rows), layer["H"], layer["I"])
    assert_close(y[rows], ref, f"T={T} rows {rows}")


def test_full_layer_prefill_256_sampled_rows():
    layer = dense_layer(1, T=256)
    _sampled(layer, 256, [0, 1, 63, 64, 127, 128, 200, 255])


def test_full_layer_prefill_2048_sampled_rows_with_outliers():
    layer = dense_layer(2, T=2048, outlier_frac=0.01)
    xf = synth.bf16_bits_to_f32(layer["x"])
    outliers = np.nonzero(np.abs(xf).max(axis=1) > 8.0)[0]
    assert len(outliers) == 20
    # the first and last row of every 256-token tile, the rows either side of
    # each tile's 128-row split between the two CTAs of a pair, every outlier row
    tiles = [r for t in range(0, 2048, 256) for r in (t, t + 127, t + 128, t + 255)]
    rows = sorted(set(tiles + [1000] + list(outliers)))
    _sampled(layer, 2048, rows)


def test_full_layer_decode_tokens():
    layer = dense_layer(3)
    Wg, Wu, Wd = dev(layer["Wg"]), dev(layer["Wu"]), dev(layer["Wd"])
    for r in range(3):
        x = layer["x"][r:r + 1].copy()
        y = zffn.swiglu_q4k(x_dev(x), Wg, Wu, Wd, layer["I"])
        assert zffn.get_device_error() == zffn.OK
        ref = orc.swiglu_ffn(x, layer["Wg"], layer["Wu"], layer["Wd"], 1, layer["H"], layer["I"])
        assert_close(y, ref, f"decode token {r}")


# ---- calls chained on one stream ----------------------------------------------

def test_chained_calls_on_one_stream_when_the_units_fill_the_gpu():
    # 2 token tiles x 38 intermediate chunks = 76 units: one per CTA pair, so
    # the prefill kernel starts while the x conversion before it runs.  A
    # plain call, then two residual calls into the same y, back to back on one
    # stream (nothing synchronises the host in between): y = 3 * block(x).
    H, I, T = 256, 9728, 512
    rng = np.random.default_rng(910)
    Wg = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wu = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wd = synth.random_q4k_blocks(rng, H, I, 1e-2)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    xd, Wgd, Wud, Wdd = x_dev(x), dev(Wg), dev(Wu), dev(Wd)
    y = zffn.swiglu_q4k(xd, Wgd, Wud, Wdd, I)
    zffn.swiglu_q4k(xd, Wgd, Wud, Wdd, I, y=y, residual=True)
    zffn.swiglu_q4k(xd, Wgd, Wud, Wdd, I, y=y, residual=True)
    assert zffn.get_device_error() == zffn.OK
    rows = [0, 1, 127, 128, 255, 256, 383, 384, 511]
    ref = orc.swiglu_ffn(x[rows].copy(), Wg, Wu, Wd, len(rows), H, I)
    assert_close(y[rows], 3.0 * ref, "three chained calls")
