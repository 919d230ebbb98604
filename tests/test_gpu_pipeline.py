"""The host pipeline (zffn_pipeline_*): blocks over host buffers with the copies
overlapped, against the oracle and against the device-buffer entry point."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_ffn_gb300 import synth, zffn
from tests.gpu_util import assert_close, dense_layer, dev, x_dev

pytestmark = pytest.mark.gpu


def pinned_bf16(bits):
    t = torch.empty(bits.shape, dtype=torch.bfloat16, pin_memory=True)
    t.view(torch.int16).copy_(torch.from_numpy(bits.astype(np.uint16).view(np.int16)))
    return t


@pytest.mark.parametrize("depth", [2, 3])
def test_pipeline_tiny_layer_many_submissions(depth):
    d = synth.tiny()
    T, H, I = d["T"], d["H"], d["I"]
    W = [dev(d[n]) for n in ("Wg", "Wu", "Wd")]
    torch.cuda.synchronize()
    rng = np.random.default_rng(depth)
    xs = [synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)) for _ in range(7)]
    ys = [torch.empty((T, H), dtype=torch.float32, pin_memory=True) for _ in xs]
    p = zffn.Pipeline(T, H, I, depth)
    try:
        for x, y in zip(xs, ys):
            p.submit(pinned_bf16(x), *W, y)
        p.sync()
    finally:
        p.close()
    assert zffn.get_device_error() == zffn.OK
    for i, (x, y) in enumerate(zip(xs, ys)):
        ref = orc.swiglu_ffn(x, d["Wg"], d["Wu"], d["Wd"], T, H, I)
        assert_close(y, ref, f"pipeline submission {i}")


def test_pipeline_single_token_rotating_weights():
    # T = 1 runs the single-token kernels; consecutive submissions alternate
    # between two layers, as consecutive layers of a decode step do
    H, I = 1024, 1472
    rng = np.random.default_rng(8)
    layers = []
    for _ in range(2):
        Wg, Wu, Wd = (synth.random_q4k_blocks(rng, I, H, 1e-2), synth.random_q4k_blocks(rng, I, H, 1e-2),
                      synth.random_q4k_blocks(rng, H, I, 1e-2))
        layers.append(((Wg, Wu, Wd), [dev(Wg), dev(Wu), dev(Wd)]))
    torch.cuda.synchronize()
    xs = [synth.f32_to_bf16_bits(rng.standard_normal((1, H)).astype(np.float32)) for _ in range(6)]
    ys = [torch.empty((1, H), dtype=torch.float32, pin_memory=True) for _ in xs]
    p = zffn.Pipeline(1, H, I, 2)
    try:
        for i, (x, y) in enumerate(zip(xs, ys)):
            p.submit(pinned_bf16(x), *layers[i % 2][1], y)
        p.sync()
    finally:
        p.close()
    assert zffn.get_device_error() == zffn.OK
    for i, (x, y) in enumerate(zip(xs, ys)):
        Wg, Wu, Wd = layers[i % 2][0]
        assert_close(y, orc.swiglu_ffn(x, Wg, Wu, Wd, 1, H, I), f"token {i}")


def test_pipeline_full_layer_matches_device_entry_point():
    L = dense_layer(1, T=256)
    T, H, I = 256, L["H"], L["I"]
    W = [dev(L[n]) for n in ("Wg", "Wu", "Wd")]
    torch.cuda.synchronize()
    rng = np.random.default_rng(9)
    xs = [synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)) for _ in range(3)]
    ys = [torch.empty((T, H), dtype=torch.float32, pin_memory=True) for _ in xs]
    p = zffn.Pipeline(T, H, I, 2)
    try:
        for x, y in zip(xs, ys):
            p.submit(pinned_bf16(x), *W, y)
        p.sync()
    finally:
        p.close()
    for x, y in zip(xs, ys):
        ref = zffn.swiglu_q4k(x_dev(x), *W, I).cpu()
        # the same kernels; only the order of the fp32 reductions into y differs
        assert torch.allclose(y, ref, rtol=1e-4, atol=1e-5)
    rows = [0, 77, 255]
    assert_close(ys[2][rows], orc.swiglu_ffn(xs[2][rows].copy(), L["Wg"], L["Wu"], L["Wd"], 3, H, I),
                 "pipeline full layer")


def test_pipeline_rejects_wrong_buffers():
    d = synth.tiny()
    W = [dev(d[n]) for n in ("Wg", "Wu", "Wd")]
    p = zffn.Pipeline(d["T"], d["H"], d["I"], 2)
    try:
        with pytest.raises(ValueError):
            p.submit(torch.empty((d["T"], d["H"] + 1), dtype=torch.bfloat16), *W,
                     torch.empty((d["T"], d["H"]), dtype=torch.float32))
        with pytest.raises(ValueError):
            p.submit(torch.empty((d["T"], d["H"]), dtype=torch.bfloat16, device="cuda"), *W,
                     torch.empty((d["T"], d["H"]), dtype=torch.float32))
    finally:
        p.close()


@pytest.mark.parametrize("T", [1, 40])
def test_pipeline_routed_block(T):
    # router on the device, then routed blocks over host buffers
    E, H, I, k = 16, 512, 384, 4
    rng = np.random.default_rng(10 + T)
    Wg = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wu = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wd = np.stack([synth.random_q4k_blocks(rng, H, I, 1e-2) for _ in range(E)])
    W = [dev(Wg), dev(Wu), dev(Wd)]
    logits = [rng.standard_normal((T, E)).astype(np.float32) for _ in range(3)]
    routes = [zffn.moe_router_topk(dev(lg), k) for lg in logits]
    torch.cuda.synchronize()
    xs = [synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)) for _ in range(3)]
    ys = [torch.empty((T, H), dtype=torch.float32, pin_memory=True) for _ in xs]
    p = zffn.Pipeline(T, H, I, 2)
    try:
        for x, (ids, w), y in zip(xs, routes, ys):
            p.submit_moe(pinned_bf16(x), ids, w, *W, E, y)
        p.sync()
    finally:
        p.close()
    assert zffn.get_device_error() == zffn.OK
    for i, (x, lg, y) in enumerate(zip(xs, logits, ys)):
        ids, w = orc.route_top_k(lg, k)
        assert_close(y, orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k), f"routed {i}")
