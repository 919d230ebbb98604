"""The device-side router (logits -> top-k expert ids -> softmax weights)
against the oracle, through the C ABI.

The ids are integer decisions taken from comparisons of the same fp32 logits
on both sides: they must match exactly.  The weights are fp32 on the GPU
(expf, a warp-wide fp32 sum, one division) and fp64 rounded once to fp32 in
the oracle: expf is within 2 ulp, the sum of at most 64 positive terms within
about 6 ulp in a tree, the division within 0.5 ulp, so a relative bound of
2e-6 (about 17 ulp) holds with margin; `atol` covers weights that fall into
the fp32 subnormal range."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_ffn_gb300 import synth, zffn
from tests.gpu_util import assert_close, dev, moe_layer, x_dev

pytestmark = pytest.mark.gpu

W_RTOL = 2e-6
W_ATOL = 1e-37


def check(logits, k):
    ids_d, w_d = zffn.moe_router_topk(dev(logits), k)
    torch.cuda.synchronize()
    ids_ref, w_ref = orc.route_top_k(logits, k)
    ids_g, w_g = ids_d.cpu().numpy(), w_d.cpu().numpy()
    assert np.array_equal(ids_g, ids_ref)
    nan = np.isnan(w_ref)
    assert np.array_equal(np.isnan(w_g), nan)
    np.testing.assert_allclose(w_g[~nan], w_ref[~nan], rtol=W_RTOL, atol=W_ATOL)
    return ids_g, w_g


def test_router_on_the_routed_layer_logits():
    # the routed layer's own logits, T=256 and T=1 (E=128, top-8, seed 4)
    for T in (256, 1):
        check(synth.MoE(T).logits, 8)


@pytest.mark.parametrize("T,E,k", [(1, 128, 8), (37, 33, 5), (9, 4096, 64), (1000, 64, 1),
                                   (3, 64, 64), (17, 1, 1), (5, 100, 33), (6, 256, 16),
                                   (11, 200, 8), (4, 257, 40), (2, 1000, 7)])
def test_router_shapes(T, E, k):
    # ragged T (blocks of 8 tokens), E not a multiple of 32, k past one warp,
    # E on both sides of the register-resident limits (128, 256)
    rng = np.random.default_rng(T * 7919 + E * 31 + k)
    check(rng.standard_normal((T, E)).astype(np.float32) * np.float32(2.0), k)


def test_router_ties_go_to_the_lower_index():
    rng = np.random.default_rng(5)
    logits = rng.integers(-3, 4, size=(512, 128)).astype(np.float32)
    ids, _ = check(logits, 8)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :8]
    assert np.array_equal(ids, order)
    # all equal: the first k indices, equal weights
    ids, w = check(np.full((4, 96), -1.5, np.float32), 6)
    assert np.array_equal(ids, np.tile(np.arange(6), (4, 1)))
    assert np.all(w == np.float32(1.0 / 6.0))


def test_router_special_values():
    nan, inf = np.float32("nan"), np.float32("inf")
    logits = np.array([[nan, -inf, 1.0, -0.0, 0.0, nan, -3.0, 2.5],
                       [-inf, -inf, -inf, 0.5, nan, 7.0, -0.0, 0.0],
                       [nan, nan, nan, nan, nan, nan, nan, nan],
                       [inf, 1.0, inf, -2.0, 0.0, 3.0, -1.0, 2.0]], np.float32)
    for k in (1, 4, 8):
        check(logits, k)


def test_router_feeds_the_routed_block():
    # logits -> device router -> routed block, against oracle router -> oracle block
    rng = np.random.default_rng(12)
    T, E, H, I, k = 24, 16, 512, 384, 4
    Wg = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wu = np.stack([synth.random_q4k_blocks(rng, I, H, 1e-2) for _ in range(E)])
    Wd = np.stack([synth.random_q4k_blocks(rng, H, I, 1e-2) for _ in range(E)])
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    ids_d, w_d = zffn.moe_router_topk(dev(logits), k)
    y = zffn.moe_swiglu_q4k(x_dev(x), ids_d, w_d, dev(Wg), dev(Wu), dev(Wd), I, E)
    assert zffn.get_device_error() == zffn.OK
    ids, w = orc.route_top_k(logits, k)
    ref = orc.moe_swiglu_ffn(x, ids, w, Wg, Wu, Wd, T, H, I, E, k)
    assert_close(y, ref, "router -> routed block")


def test_router_full_routed_layer_ids_match_inputs_of_moe_tests():
    # the cached routed-layer fixture takes its ids from the oracle's router:
    # the device router must produce the same buffers from the same logits
    m = moe_layer(256)
    ids_d, w_d = zffn.moe_router_topk(dev(m["logits"]), m["k"])
    assert np.array_equal(ids_d.cpu().numpy(), m["ids"])
    np.testing.assert_allclose(w_d.cpu().numpy(), m["w"], rtol=W_RTOL, atol=W_ATOL)


@pytest.mark.parametrize("T,E,k", [(0, 8, 2), (4, 0, 1), (4, 5000, 8), (4, 8, 0), (4, 8, 9),
                                   (4, 128, 65)])
def test_router_rejects_bad_sizes(T, E, k):
    logits = torch.zeros((max(T, 1), max(E, 1)), dtype=torch.float32, device="cuda")
    ids = torch.zeros((max(T, 1), max(k, 1)), dtype=torch.int32, device="cuda")
    w = torch.zeros((max(T, 1), max(k, 1)), dtype=torch.float32, device="cuda")
    st = zffn.load().zffn_moe_router_topk(logits.data_ptr(), ids.data_ptr(), w.data_ptr(),
                                           T, E, k, None)
    assert st == zffn.ERR_INVALID_ARG
