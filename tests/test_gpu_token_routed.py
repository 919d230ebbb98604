"""The routed single-token layer on both of its paths, through the C ABI,
against the oracle: the one cooperative launch (every block asks for all of
its weights at once, a grid barrier between the gate/up and the down step)
and the two-kernel pair.  Shapes cover the full routed layer of the pages'
MoE workload (E=128, H=2048, I=768, top-8), blocks whose gate/up rows span
two expert slots, widths that are not a multiple of 256, many slots, invalid
and repeated slots, a per-expert down scale with accumulation, long runs of
calls (the barrier's state carries from one call to the next), and a layer
too large for the one-launch path (it falls back to the pair)."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_ffn_gb300 import synth, zffn
from tests.gpu_util import assert_close, dev, moe_layer, x_dev

pytestmark = pytest.mark.gpu


def experts(rng, E, H, I):
    Wg = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wu = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wd = np.stack([synth.random_q4k_blocks(rng, H, I, 1e-2) for _ in range(E)])
    return Wg, Wu, Wd


def token(rng, H):
    return synth.f32_to_bf16_bits(rng.standard_normal((1, H)).astype(np.float32))


class token_kernel:
    def __init__(self, v):
        self.v = v

    def __enter__(self):
        self.old = zffn.set_option(zffn.OPT_TOKEN_KERNEL, self.v)

    def __exit__(self, *exc):
        zffn.set_option(zffn.OPT_TOKEN_KERNEL, self.old)


@pytest.mark.parametrize("path", [0, 1])
def test_full_routed_layer_every_output(path):
    m = moe_layer(1)
    with token_kernel(path):
        y = zffn.moe_swiglu_q4k(x_dev(m["x"]), dev(m["ids"]), dev(m["w"]), dev(m["Wg"]), dev(m["Wu"]),
                                dev(m["Wd"]), m["I"], m["E"])
        assert zffn.get_device_error() == zffn.OK
    ref = orc.moe_swiglu_ffn(m["x"], m["ids"], m["w"], m["Wg"], m["Wu"], m["Wd"], 1, m["H"], m["I"], m["E"],
                             m["k"])
    assert_close(y, ref, f"routed T=1, path {path}")


@pytest.mark.parametrize("path", [0, 1])
@pytest.mark.parametrize("E,H,I,k", [(16, 512, 384, 4), (8, 256, 64, 2), (24, 1024, 1472, 6),
                                     (32, 4096, 512, 8), (80, 256, 128, 64)])
def test_routed_token_shapes(path, E, H, I, k):
    rng = np.random.default_rng(900 + E + H + I + k + path)
    Wg, Wu, Wd = experts(rng, E, H, I)
    ids, w = orc.route_top_k(rng.standard_normal((1, E)).astype(np.float32), k)
    ids[0, k - 1] = -1                          # an invalid slot contributes nothing
    if k > 2:
        ids[0, 1] = ids[0, 0]                   # the same expert in two slots
    x = token(rng, H)
    with token_kernel(path):
        y = zffn.moe_swiglu_q4k(x_dev(x), dev(ids), dev(w), dev(Wg), dev(Wu), dev(Wd), I, E)
        assert zffn.get_device_error() == zffn.OK
    assert_close(y, orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, 1, H, I, E, k), f"E={E} H={H} I={I} k={k}")


def test_one_launch_scale_accumulate_and_long_runs():
    # a per-expert down scale with accumulation, then 300 calls in a row with
    # different tokens and routes: each must match the oracle
    E, H, I, k = 32, 1024, 768, 8
    rng = np.random.default_rng(950)
    Wg, Wu, Wd = experts(rng, E, H, I)
    dWg, dWu, dWd = dev(Wg), dev(Wu), dev(Wd)
    scale = rng.uniform(0.25, 2.0, E).astype(np.float32)
    with token_kernel(0):
        ids, w = orc.route_top_k(rng.standard_normal((1, E)).astype(np.float32), k)
        x = token(rng, H)
        y0 = torch.full((1, H), 0.5, dtype=torch.float32, device="cuda")
        zffn.moe_swiglu_q4k_scaled(x_dev(x), dev(ids), dev(w), dev(scale), dWg, dWu, dWd, I, E, y=y0,
                                   accumulate=True)
        assert zffn.get_device_error() == zffn.OK
        ref = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, 1, H, I, E, k, down_scale=scale)
        assert_close(y0, ref + 0.5, "scale + accumulate")
        n = 300
        xs = [token(rng, H) for _ in range(n)]
        routes = [orc.route_top_k(rng.standard_normal((1, E)).astype(np.float32), k) for _ in range(n)]
        outs = [torch.empty((1, H), dtype=torch.float32, device="cuda") for _ in range(n)]
        dx = [x_dev(v) for v in xs]
        dr = [(dev(i), dev(ww)) for i, ww in routes]
        for j in range(n):
            zffn.moe_swiglu_q4k(dx[j], dr[j][0], dr[j][1], dWg, dWu, dWd, I, E, y=outs[j])
        torch.cuda.synchronize()
        assert zffn.get_device_error() == zffn.OK
    for j in list(range(0, n, 37)) + [n - 1]:
        ref = orc.moe_swiglu_ffn(xs[j], routes[j][0], routes[j][1], Wg, Wu, Wd, 1, H, I, E, k)
        assert_close(outs[j], ref, f"call {j} of {n}")


def test_launch_count_query():
    # the pages' routed layer takes the one launch; forced, or too large, the pair
    assert zffn.single_token_launches(2048, 768, 128, 8) == 1
    with token_kernel(1):
        assert zffn.single_token_launches(2048, 768, 128, 8) == 2
    assert zffn.single_token_launches(4096, 11008, 2, 2) == 2


def test_layer_too_large_for_one_launch_falls_back():
    # two experts of the dense workload's size: a block's share of the gate/up
    # rows (about 145 row pairs of 2 x 2304 bytes) exceeds its shared memory
    E, H, I, k = 2, 4096, 11008, 2
    rng = np.random.default_rng(960)
    Wg, Wu, Wd = experts(rng, E, H, I)
    ids = np.array([[1, 0]], dtype=np.int32)
    w = np.array([[0.7, 0.3]], dtype=np.float32)
    x = token(rng, H)
    with token_kernel(0):
        y = zffn.moe_swiglu_q4k(x_dev(x), dev(ids), dev(w), dev(Wg), dev(Wu), dev(Wd), I, E)
        assert zffn.get_device_error() == zffn.OK
    assert_close(y, orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, 1, H, I, E, k), "fallback to the pair")


def test_timeout_report_resets_the_barrier_and_the_path_still_works():
    # a reported timeout (here from the bounded-wait self test) resets the
    # one-launch path's barrier count; calls before and after stay correct
    E, H, I, k = 16, 512, 384, 4
    rng = np.random.default_rng(980)
    Wg, Wu, Wd = experts(rng, E, H, I)
    dW = [dev(Wg), dev(Wu), dev(Wd)]
    with token_kernel(0):
        for call in range(3):
            ids, w = orc.route_top_k(rng.standard_normal((1, E)).astype(np.float32), k)
            x = token(rng, H)
            y = zffn.moe_swiglu_q4k(x_dev(x), dev(ids), dev(w), *dW, I, E)
            assert zffn.get_device_error() == zffn.OK
            assert_close(y, orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, 1, H, I, E, k), f"call {call}")
            if call == 0:
                zffn.selftest_wait_timeout(2_000_000)
                assert zffn.get_device_error() == zffn.ERR_TIMEOUT
