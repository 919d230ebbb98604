"""Routed (mixture-of-experts) SwiGLU block on the GPU against the oracle."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_ffn_gb300 import synth, zffn
from tests.gpu_util import assert_close, dev, moe_layer, x_dev

pytestmark = pytest.mark.gpu


def experts(seed, E, H, I, dscale=1e-2):
    rng = np.random.default_rng(seed)
    Wg = np.stack([synth.random_q4k_blocks(rng, I, H, dscale) for _ in range(E)])
    Wu = np.stack([synth.random_q4k_blocks(rng, I, H, dscale) for _ in range(E)])
    Wd = np.stack([synth.random_q4k_blocks(rng, H, I, dscale) for _ in range(E)])
    return Wg, Wu, Wd


def routing(seed, T, E, k):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    return orc.route_top_k(logits, k)


def run(x, ids, w, Wg, Wu, Wd, I, E, matvec_max_t=None):
    old = None
    if matvec_max_t is not None:
        old = zffn.set_option(zffn.OPT_MATVEC_MAX_T, matvec_max_t)
    try:
        y = zffn.moe_swiglu_q4k(x_dev(x), dev(ids), dev(w), dev(Wg), dev(Wu), dev(Wd), I, E)
        assert zffn.get_device_error() == zffn.OK
    finally:
        if old is not None:
            zffn.set_option(zffn.OPT_MATVEC_MAX_T, old)
    return y


@pytest.mark.parametrize("T,E,H,I,k", [(40, 8, 512, 384, 2), (300, 16, 256, 704, 4),
                                       (5, 32, 1024, 256, 8), (1, 8, 512, 384, 2)])
def test_small_moe_tensor_core_path(T, E, H, I, k):
    Wg, Wu, Wd = experts(T + E, E, H, I)
    ids, w = routing(T * E, T, E, k)
    x = synth.f32_to_bf16_bits(np.random.default_rng(9).standard_normal((T, H)).astype(np.float32))
    y = run(x, ids, w, Wg, Wu, Wd, I, E, matvec_max_t=0)
    ref = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k)
    assert_close(y, ref, f"moe tc T={T} E={E}")


@pytest.mark.parametrize("E,H,I,k", [(8, 512, 384, 2), (16, 256, 704, 8)])
def test_small_moe_single_token_path(E, H, I, k):
    Wg, Wu, Wd = experts(E + 1, E, H, I)
    ids, w = routing(E + 2, 1, E, k)
    x = synth.f32_to_bf16_bits(np.random.default_rng(3).standard_normal((1, H)).astype(np.float32))
    y = run(x, ids, w, Wg, Wu, Wd, I, E, matvec_max_t=1)
    ref = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, 1, H, I, E, k)
    assert_close(y, ref, "moe matvec")


@pytest.mark.parametrize("path", [0, 1])
def test_invalid_ids_contribute_nothing(path):
    T = 1 if path else 20
    E, H, I, k = 6, 256, 256, 3
    Wg, Wu, Wd = experts(11, E, H, I)
    ids, w = routing(12, T, E, k)
    ids[0, 1] = -3
    ids[-1, 2] = E + 5
    x = synth.f32_to_bf16_bits(np.random.default_rng(4).standard_normal((T, H)).astype(np.float32))
    y = run(x, ids, w, Wg, Wu, Wd, I, E, matvec_max_t=path)
    ref = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k)
    assert_close(y, ref, "invalid ids")


def test_single_expert_routing_equals_dense_call():
    T, E, H, I = 70, 4, 512, 384
    Wg, Wu, Wd = experts(21, E, H, I)
    ids = np.full((T, 1), 2, dtype=np.int32)
    w = np.ones((T, 1), dtype=np.float32)
    x = synth.f32_to_bf16_bits(np.random.default_rng(5).standard_normal((T, H)).astype(np.float32))
    y = run(x, ids, w, Wg, Wu, Wd, I, E, matvec_max_t=0)
    y_dense = zffn.swiglu_q4k(x_dev(x), dev(Wg[2]), dev(Wu[2]), dev(Wd[2]), I)
    torch.cuda.synchronize()
    ref = orc.swiglu_ffn(x, Wg[2], Wu[2], Wd[2], T, H, I)
    assert_close(y, ref, "moe k=1")
    assert_close(y_dense, ref, "dense")


def test_full_moe_config_single_token():
    m = moe_layer(1)
    y = run(m["x"], m["ids"], m["w"], m["Wg"], m["Wu"], m["Wd"], m["I"], m["E"])
    ref = orc.moe_swiglu_ffn(m["x"], m["ids"], m["w"], m["Wg"], m["Wu"], m["Wd"], 1, m["H"],
                             m["I"], m["E"], m["k"])
    assert_close(y, ref, "moe T=1")


def test_full_moe_config_256_tokens_sampled_rows():
    m = moe_layer(256)
    y = run(m["x"], m["ids"], m["w"], m["Wg"], m["Wu"], m["Wd"], m["I"], m["E"])
    rows = list(range(0, 256, 16)) + [1, 17, 127, 128, 129, 255]
    ref = orc.moe_swiglu_ffn(m["x"][rows].copy(), m["ids"][rows].copy(), m["w"][rows].copy(),
                             m["Wg"], m["Wu"], m["Wd"], len(rows), m["H"], m["I"], m["E"], m["k"])
    assert_close(y[rows], ref, "moe T=256 sampled")


@pytest.mark.parametrize("T,path,fmt", [(1, 1, zffn.FMT_Q4_K), (37, 0, zffn.FMT_Q4_K),
                                        (1, 1, zffn.FMT_Q5_K), (1, 1, zffn.FMT_Q5_1), (1, 1, zffn.FMT_Q6_K)])
def test_per_expert_down_scale(T, path, fmt):
    # a scale on each expert's down projection, applied inside the routed call
    E, H, I, k = 8, 512, 384, 3
    rng = np.random.default_rng(77 + T + fmt)
    Wg = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wu = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wd = np.stack([synth.random_blocks(rng, fmt, H, I, 1e-2) for _ in range(E)])
    ids, w = routing(31 + T, T, E, k)
    ids[0, 2] = -1                       # an invalid slot still contributes nothing
    scale = np.array([1.5, -0.25, 0.0, 2.0, 0.75, 1.0, -3.0, 0.125], dtype=np.float32)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    ref = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k, wd_fmt=fmt, down_scale=scale)
    old = zffn.set_option(zffn.OPT_MATVEC_MAX_T, path)
    try:
        y = zffn.moe_swiglu_q4k_scaled(x_dev(x), dev(ids), dev(w), dev(scale), dev(Wg), dev(Wu),
                                       dev(Wd), I, E, wd_fmt=fmt)
        assert zffn.get_device_error() == zffn.OK
        assert_close(y, ref, f"down scale T={T} fmt={fmt}")
        # accumulate: y0 + the scaled block
        y0 = torch.full((T, H), 0.5, dtype=torch.float32, device="cuda")
        zffn.moe_swiglu_q4k_scaled(x_dev(x), dev(ids), dev(w), dev(scale), dev(Wg), dev(Wu), dev(Wd),
                                   I, E, wd_fmt=fmt, y=y0, accumulate=True)
        assert zffn.get_device_error() == zffn.OK
        assert_close(y0, ref + 0.5, f"down scale accumulate T={T} fmt={fmt}")
        # no scale equals the unscaled call
        y1 = zffn.moe_swiglu_q4k_scaled(x_dev(x), dev(ids), dev(w), None, dev(Wg), dev(Wu), dev(Wd),
                                        I, E, wd_fmt=fmt)
        assert zffn.get_device_error() == zffn.OK
        assert_close(y1, orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k, wd_fmt=fmt),
                     f"no scale T={T} fmt={fmt}")
    finally:
        zffn.set_option(zffn.OPT_MATVEC_MAX_T, old)


def test_per_expert_down_scale_full_config_256_tokens():
    m = moe_layer(256)
    scale = np.random.default_rng(8).uniform(0.5, 2.0, m["E"]).astype(np.float32)
    y = zffn.moe_swiglu_q4k_scaled(x_dev(m["x"]), dev(m["ids"]), dev(m["w"]), dev(scale), dev(m["Wg"]),
                                   dev(m["Wu"]), dev(m["Wd"]), m["I"], m["E"])
    assert zffn.get_device_error() == zffn.OK
    rows = list(range(0, 256, 32)) + [255]
    ref = orc.moe_swiglu_ffn(m["x"][rows].copy(), m["ids"][rows].copy(), m["w"][rows].copy(),
                             m["Wg"], m["Wu"], m["Wd"], len(rows), m["H"], m["I"], m["E"], m["k"],
                             down_scale=scale)
    assert_close(y[rows], ref, "moe T=256 down scale")


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("T,E,H,I,k", [(40, 8, 512, 384, 2), (300, 16, 256, 704, 4), (5, 32, 1024, 256, 8),
                                       (64, 4, 256, 2048, 3), (200, 3, 512, 192, 2), (1, 8, 512, 384, 2)])
def test_both_routed_tensor_core_kernels(kernel, T, E, H, I, k):
    # kernel 1: groups of 32 rows of one expert, weights on the MMA's M side;
    # kernel 2: 128-row expert tiles on the prefill kernel.  Shapes cover a
    # partial last W_down block (I = 704, 192), several intermediate chunks
    # (I = 2048), experts with more than one group (T * k / E = 200).
    Wg, Wu, Wd = experts(T + 3 * E + I, E, H, I)
    ids, w = routing(T * E + k, T, E, k)
    x = synth.f32_to_bf16_bits(np.random.default_rng(T + I).standard_normal((T, H)).astype(np.float32))
    old = zffn.set_option(zffn.OPT_MOE_KERNEL, kernel)
    try:
        y = run(x, ids, w, Wg, Wu, Wd, I, E, matvec_max_t=0)
    finally:
        zffn.set_option(zffn.OPT_MOE_KERNEL, old)
    ref = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k)
    assert_close(y, ref, f"routed kernel {kernel} T={T} E={E} H={H} I={I} k={k}")


@pytest.mark.parametrize("kernel", [1, 2])
def test_both_routed_kernels_full_config_256_tokens(kernel):
    m = moe_layer(256)
    old = zffn.set_option(zffn.OPT_MOE_KERNEL, kernel)
    try:
        y = run(m["x"], m["ids"], m["w"], m["Wg"], m["Wu"], m["Wd"], m["I"], m["E"])
    finally:
        zffn.set_option(zffn.OPT_MOE_KERNEL, old)
    rows = list(range(0, 256, 16)) + [1, 17, 127, 128, 129, 255]
    ref = orc.moe_swiglu_ffn(m["x"][rows].copy(), m["ids"][rows].copy(), m["w"][rows].copy(),
                             m["Wg"], m["Wu"], m["Wd"], len(rows), m["H"], m["I"], m["E"], m["k"])
    assert_close(y[rows], ref, f"moe T=256 kernel {kernel}")


def test_chained_routed_calls_on_one_stream():
    # routing, gather and the grouped kernel of one call are chained by
    # programmatic dependent launch; a plain call and two residual calls into
    # the same y, back to back on one stream, give 3 times the block
    E, H, I, k, T = 16, 512, 768, 4, 96
    Wg, Wu, Wd = experts(930, E, H, I)
    ids, w = routing(931, T, E, k)
    x = synth.f32_to_bf16_bits(np.random.default_rng(932).standard_normal((T, H)).astype(np.float32))
    args = (x_dev(x), dev(ids), dev(w), dev(Wg), dev(Wu), dev(Wd), I, E)
    y = zffn.moe_swiglu_q4k(*args)
    zffn.moe_swiglu_q4k(*args, y=y, residual=True)
    zffn.moe_swiglu_q4k(*args, y=y, residual=True)
    assert zffn.get_device_error() == zffn.OK
    ref = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k)
    assert_close(y, 3.0 * ref, "three chained routed calls")
