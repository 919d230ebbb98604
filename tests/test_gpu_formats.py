"""Other block formats of W_down (Q5_K, Q6_K, Q5_1) on the GPU through the C
ABI: the dequantisation bit-exact against the oracle, and the single-token
dense and routed blocks with W_down in each format against the oracle at the
block's tolerance."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_ffn_gb300 import synth, zffn
from tests.gpu_util import assert_close, dev, x_dev

pytestmark = pytest.mark.gpu

FORMATS = [zffn.FMT_Q5_K, zffn.FMT_Q6_K, zffn.FMT_Q5_1]


@pytest.mark.parametrize("fmt", FORMATS + [zffn.FMT_Q4_K])
@pytest.mark.parametrize("rows,cols", [(64, 768), (7, 11008), (33, 704)])
def test_dequant_bit_exact(fmt, rows, cols):
    rng = np.random.default_rng(fmt * 100 + rows)
    blocks = synth.random_blocks(rng, fmt, rows, cols, 1e-2)
    got = zffn.dequant_fmt(dev(blocks), fmt, rows, cols).cpu().numpy()
    ref = orc.dequant_fmt(blocks, fmt, rows, cols)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def token(rng, H):
    return synth.f32_to_bf16_bits(rng.standard_normal((1, H)).astype(np.float32))


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("H,I", [(1024, 1472), (256, 704), (4096, 11008)])
def test_single_token_block(fmt, H, I):
    rng = np.random.default_rng(fmt + H + I)
    Wg = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wu = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wd = synth.random_blocks(rng, fmt, H, I, 1e-2)
    x = token(rng, H)
    y = zffn.swiglu_q4k_wd(x_dev(x), dev(Wg), dev(Wu), dev(Wd), fmt, I)
    assert zffn.get_device_error() == zffn.OK
    assert_close(y, orc.swiglu_ffn(x, Wg, Wu, Wd, 1, H, I, wd_fmt=fmt), f"fmt {fmt} H={H} I={I}")


def offset_copy(a, offset):
    """a (uint8) on the device, starting `offset` bytes past a 16-byte boundary."""
    buf = torch.zeros(a.nbytes + 32, dtype=torch.uint8, device="cuda")
    assert buf.data_ptr() % 16 == 0
    out = buf[offset:offset + a.nbytes]
    out.copy_(torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8)).cuda())
    return out


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("H,I,wd_offset", [(256, 64, 4), (512, 192, 0), (768, 320, 8), (1024, 1472, 4),
                                           (4096, 11008, 12)])
def test_single_token_block_short_rows_and_unaligned_wd(fmt, H, I, wd_offset):
    # rows of fewer than four 256-weight units (several output rows in one
    # pass of a warp), and W_down 4, 8 or 12 bytes past a 16-byte boundary
    # (copied in 4-byte words instead of 16-byte pieces)
    rng = np.random.default_rng(600 + fmt + H + I + wd_offset)
    Wg = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wu = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wd = synth.random_blocks(rng, fmt, H, I, 1e-2)
    x = token(rng, H)
    Wd_dev = offset_copy(Wd, wd_offset)
    y = zffn.swiglu_q4k_wd(x_dev(x), dev(Wg), dev(Wu), Wd_dev, fmt, I)
    assert zffn.get_device_error() == zffn.OK
    assert_close(y, orc.swiglu_ffn(x, Wg, Wu, Wd, 1, H, I, wd_fmt=fmt), f"fmt {fmt} H={H} I={I} +{wd_offset}")


@pytest.mark.parametrize("fmt", FORMATS)
def test_routed_single_token_unaligned_wd_and_no_valid_slot(fmt):
    # every expert's W_down 4 bytes past a 16-byte boundary, slots in any
    # order with repeats; then a token whose slots are all invalid: y = 0, or
    # y unchanged when accumulating
    E, H, I, k = 6, 512, 320, 5
    rng = np.random.default_rng(700 + fmt)
    Wg = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wu = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wd = np.stack([synth.random_blocks(rng, fmt, H, I, 1e-2) for _ in range(E)])
    ids = np.array([[5, 0, 5, -1, 2]], dtype=np.int32)
    w = rng.uniform(0.1, 1.0, (1, k)).astype(np.float32)
    x = token(rng, H)
    Wd_dev = offset_copy(Wd, 4)
    y = zffn.moe_swiglu_q4k_wd(x_dev(x), dev(ids), dev(w), dev(Wg), dev(Wu), Wd_dev, fmt, I, E)
    assert zffn.get_device_error() == zffn.OK
    assert_close(y, orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, 1, H, I, E, k, wd_fmt=fmt), f"routed fmt {fmt} +4")
    bad = np.array([[-1, E, E + 7, -3, 99]], dtype=np.int32)
    y = zffn.moe_swiglu_q4k_wd(x_dev(x), dev(bad), dev(w), dev(Wg), dev(Wu), Wd_dev, fmt, I, E)
    assert zffn.get_device_error() == zffn.OK
    assert torch.count_nonzero(y).item() == 0
    y0 = torch.full((1, H), 0.25, dtype=torch.float32, device="cuda")
    zffn.moe_swiglu_q4k_scaled(x_dev(x), dev(bad), dev(w), None, dev(Wg), dev(Wu), Wd_dev, I, E, wd_fmt=fmt,
                               y=y0, accumulate=True)
    assert zffn.get_device_error() == zffn.OK
    assert torch.all(y0 == 0.25).item()


@pytest.mark.parametrize("fmt", FORMATS)
def test_routed_single_token_full_config(fmt):
    # E = 128, H = 2048, I = 768, top-8 with every expert's W_down in fmt
    E, H, I, k = 128, 2048, 768, 8
    rng = np.random.default_rng(200 + fmt)
    Wg = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wu = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wd = np.stack([synth.random_blocks(rng, fmt, H, I, 1e-2) for _ in range(E)])
    ids, w = orc.route_top_k(rng.standard_normal((1, E)).astype(np.float32), k)
    ids[0, 3] = E + 2                       # an invalid slot contributes nothing
    x = token(rng, H)
    y = zffn.moe_swiglu_q4k_wd(x_dev(x), dev(ids), dev(w), dev(Wg), dev(Wu), dev(Wd), fmt, I, E)
    assert zffn.get_device_error() == zffn.OK
    ref = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, 1, H, I, E, k, wd_fmt=fmt)
    assert_close(y, ref, f"routed fmt {fmt}")


def test_q4k_format_code_is_the_regular_block():
    rng = np.random.default_rng(300)
    H, I = 512, 384
    W = [synth.random_q4k_blocks(rng, I, H, 1e-2), synth.random_q4k_blocks(rng, I, H, 1e-2),
         synth.random_q4k_blocks(rng, H, I, 1e-2)]
    x = synth.f32_to_bf16_bits(rng.standard_normal((5, H)).astype(np.float32))
    y = zffn.swiglu_q4k_wd(x_dev(x), *[dev(a) for a in W], zffn.FMT_Q4_K, I)
    assert_close(y, orc.swiglu_ffn(x, *W, 5, H, I), "Q4_K through the format entry")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("T,H,I", [(2, 256, 704), (33, 1024, 1472), (100, 512, 384), (40, 256, 2048)])
def test_several_tokens_dense(fmt, T, H, I):
    # T > 1: the grouped tensor-core kernel (groups of 32 tokens); shapes with a
    # partial last block (704, 1472, 384), a group boundary (33), several
    # groups (100), several intermediate chunks (2048)
    rng = np.random.default_rng(400 + fmt + T + I)
    Wg = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wu = synth.random_q4k_blocks(rng, I, H, 1e-2)
    Wd = synth.random_blocks(rng, fmt, H, I, 1e-2)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    y = zffn.swiglu_q4k_wd(x_dev(x), dev(Wg), dev(Wu), dev(Wd), fmt, I)
    assert zffn.get_device_error() == zffn.OK
    assert_close(y, orc.swiglu_ffn(x, Wg, Wu, Wd, T, H, I, wd_fmt=fmt), f"fmt {fmt} T={T} H={H} I={I}")


@pytest.mark.parametrize("fmt", FORMATS)
def test_several_tokens_routed_full_config(fmt):
    # E = 128, H = 2048, I = 768, top-8, T = 64, every expert's W_down in fmt,
    # with a per-expert down scale and an invalid slot
    E, H, I, k, T = 128, 2048, 768, 8, 64
    rng = np.random.default_rng(500 + fmt)
    Wg = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wu = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wd = np.stack([synth.random_blocks(rng, fmt, H, I, 1e-2) for _ in range(E)])
    ids, w = orc.route_top_k(rng.standard_normal((T, E)).astype(np.float32), k)
    ids[5, 2] = -1
    scale = rng.uniform(0.5, 1.5, E).astype(np.float32)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    y = zffn.moe_swiglu_q4k_scaled(x_dev(x), dev(ids), dev(w), dev(scale), dev(Wg), dev(Wu), dev(Wd), I, E,
                                   wd_fmt=fmt)
    assert zffn.get_device_error() == zffn.OK
    rows = [0, 5, 31, 32, 63]
    ref = orc.moe_swiglu_ffn(x[rows].copy(), ids[rows].copy(), w[rows].copy(), Wg, Wu, Wd, len(rows), H, I, E,
                             k, wd_fmt=fmt, down_scale=scale)
    assert_close(y[rows], ref, f"routed T=64 fmt {fmt}")


def test_small_format_call_then_larger_q4k_single_token():
    # the gate/up kernel is shared by both single-token paths: a format call at
    # a small width must not leave it a shared-memory limit that a later, wider
    # Q4_K call exceeds
    rng = np.random.default_rng(302)
    H, I = 256, 256
    small = [dev(synth.random_q4k_blocks(rng, I, H, 1e-2)), dev(synth.random_q4k_blocks(rng, I, H, 1e-2)),
             dev(synth.random_blocks(rng, zffn.FMT_Q5_K, H, I, 1e-2))]
    zffn.swiglu_q4k_wd(x_dev(token(rng, H)), *small, zffn.FMT_Q5_K, I)
    H, I = 8192, 1024
    W = [synth.random_q4k_blocks(rng, I, H, 1e-2), synth.random_q4k_blocks(rng, I, H, 1e-2),
         synth.random_q4k_blocks(rng, H, I, 1e-2)]
    x = token(rng, H)
    y = zffn.swiglu_q4k(x_dev(x), *[dev(a) for a in W], I)
    assert zffn.get_device_error() == zffn.OK
    assert_close(y, orc.swiglu_ffn(x, *W, 1, H, I), "Q4_K single token after a format call")
