"""Shared helpers of the GPU parity tests: upload, tolerance check, cached
full-size workloads (inputs from quantized_ffn_gb300.synth, Q4_K made by the
oracle's quantiser, expected values from the oracle)."""
import functools

import numpy as np
import torch

from oracle import oracle as orc
from quantized_ffn_gb300 import synth

# Parity bar of the block: max|y - y_ref| / max|y_ref| <= 1e-2 and relative L2 <= 5e-3.
MAX_REL = 1e-2
L2_REL = 5e-3


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.array(a, copy=True, order="C")).cuda()
    return t if dtype is None else t.view(dtype)


def x_dev(x_bits: np.ndarray) -> torch.Tensor:
    return dev(x_bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16)


def assert_close(y_gpu: torch.Tensor, y_ref: np.ndarray, what: str = ""):
    y = y_gpu.detach().float().cpu().numpy().astype(np.float64)
    ref = np.asarray(y_ref, dtype=np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    peak = np.abs(ref).max()
    if peak == 0.0:
        assert np.abs(y).max() <= 1e-6, f"{what}: expected zeros, got {np.abs(y).max()}"
        return
    max_rel = np.abs(y - ref).max() / peak
    l2 = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert max_rel <= MAX_REL and l2 <= L2_REL, f"{what}: max_rel={max_rel:.3e} l2={l2:.3e}"
    return max_rel, l2


@functools.lru_cache(maxsize=None)
def dense_layer(seed: int, H: int = 4096, I: int = 11008, T: int = 0, outlier_frac: float = 0.0):
    """Q4_K layer (oracle quantiser) + bf16 activations of a synth workload."""
    if T:
        d = synth.prefill(T, seed, H, I, outlier_frac)
    else:
        d = synth.decode(n_tokens=8, seed=seed, H=H, I=I)
    Wg = orc.q4k_quantize(d["Wg_f32"])
    Wu = orc.q4k_quantize(d["Wu_f32"])
    Wd = orc.q4k_quantize(d["Wd_f32"])
    return dict(x=d["x"], Wg=Wg, Wu=Wu, Wd=Wd, H=H, I=I)


@functools.lru_cache(maxsize=None)
def moe_layer(T: int, E: int = 128, H: int = 2048, I: int = 768, top_k: int = 8, seed: int = 4):
    m = synth.MoE(T, seed=seed, E=E, H=H, I=I, top_k=top_k)
    Wg = np.empty((E, I, synth.row_bytes(H)), np.uint8)
    Wu = np.empty_like(Wg)
    Wd = np.empty((E, H, synth.row_bytes(I)), np.uint8)
    for e in range(E):
        g, u, d = m.expert_f32(e)
        Wg[e] = orc.q4k_quantize(g)
        Wu[e] = orc.q4k_quantize(u)
        Wd[e] = orc.q4k_quantize(d)
    ids, w = orc.route_top_k(m.logits, top_k)
    return dict(x=m.x, logits=m.logits, ids=ids, w=w, Wg=Wg, Wu=Wu, Wd=Wd, E=E, H=H, I=I, k=top_k)
