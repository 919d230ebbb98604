"""Q4_K unpack and quantiser on the GPU: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_ffn_gb300 import synth, zffn
from tests.gpu_util import dev
from tests.q4k_blocks import make_block

pytestmark = pytest.mark.gpu


def _dequant(blocks_np, rows, cols):
    out = zffn.q4k_dequant(dev(blocks_np), rows, cols)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_dequant_tiny_config_matrices_bit_exact():
    t = synth.tiny()
    for W, rows, cols in ((t["Wg"], 704, 256), (t["Wd"], 256, 704)):
        got = _dequant(W, rows, cols)
        want = orc.q4k_dequant(W, rows, cols)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_dequant_million_random_blocks_bit_exact():
    rng = np.random.default_rng(123)
    rows, cols = 4096, 65536           # 1,048,576 blocks
    W = synth.random_q4k_blocks(rng, rows, cols, dscale=0.5)
    got = _dequant(W, rows, cols)
    want = orc.q4k_dequant(W, rows, cols)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_dequant_every_code_scale_min_bit_exact():
    q = [(k % 32) % 16 for k in range(256)]
    pairs = [(s, m) for s in range(64) for m in range(64)]
    blocks = []
    for d, dmin in ((0.000123, 0.00456), (2.0 ** -24, 3 * 2.0 ** -24), (65504.0, 0.5)):
        for i in range(0, len(pairs), 8):
            blocks.append(make_block(d, dmin, [p[0] for p in pairs[i:i + 8]],
                                     [p[1] for p in pairs[i:i + 8]], q))
    W = np.frombuffer(b"".join(blocks), dtype=np.uint8).reshape(len(blocks), 144)
    got = _dequant(W, len(blocks), 256)
    want = orc.q4k_dequant(W, len(blocks), 256)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("rows,cols,scale", [(512, 4096, 0.02), (7, 300, 1.0), (64, 11008, 0.02),
                                             (3, 768, 1e-6), (5, 256, 3e3)])
def test_quantize_matches_oracle_bytes(rows, cols, scale):
    rng = np.random.default_rng(rows * 7 + cols)
    w = (rng.standard_normal((rows, cols)) * scale).astype(np.float32)
    w[0, :17] = 0.0
    if rows > 2:
        w[2] = np.abs(w[2])            # an all-non-negative row
    got = zffn.q4k_quantize(dev(w))
    torch.cuda.synchronize()
    want = orc.q4k_quantize(w)
    assert np.array_equal(got.cpu().numpy(), want)


def test_quantize_zero_rows():
    w = np.zeros((4, 512), dtype=np.float32)
    got = zffn.q4k_quantize(dev(w)).cpu().numpy()
    assert not got.any()
