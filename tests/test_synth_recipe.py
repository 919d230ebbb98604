"""The seeded input generators keep the recipe they state: the same seed gives
the same bytes, the outlier rows are the stated share scaled by the stated
factor, the block generators fill the fp16 scale fields with finite values of
the stated sign and leave every other byte uniform, and each expert of the
routed workload comes from its own stream whatever the token count."""
import numpy as np

from quantized_ffn_gb300 import synth


def test_same_seed_same_bytes():
    a, b = synth.prefill(64, seed=2, H=256, I=512, outlier_frac=0.05), \
        synth.prefill(64, seed=2, H=256, I=512, outlier_frac=0.05)
    for k in ("x", "Wg_f32", "Wu_f32", "Wd_f32"):
        assert np.array_equal(a[k], b[k]), k
    c = synth.prefill(64, seed=3, H=256, I=512, outlier_frac=0.05)
    assert not np.array_equal(a["x"], c["x"])
    assert np.array_equal(synth.tiny()["Wd"], synth.tiny()["Wd"])


def test_outlier_rows_are_the_stated_share_and_scale():
    T, H = 2048, 1024
    d = synth.prefill(T, seed=2, H=H, I=256, outlier_frac=0.01)
    x = synth.bf16_bits_to_f32(d["x"]).astype(np.float64)
    rms = np.sqrt((x * x).mean(axis=1))
    big = rms > 5.0
    assert big.sum() == round(0.01 * T) == 20
    # scaled rows: N(0, 20^2); the rest N(0, 1)
    assert abs(rms[big].mean() - 20.0) < 1.0 and abs(rms[~big].mean() - 1.0) < 0.05
    w = d["Wg_f32"].astype(np.float64)
    assert abs(w.std() - 0.02) < 1e-3 and abs(w.mean()) < 1e-3


def _fp16_field(blocks, rows, nb, bb, off):
    return blocks.reshape(rows, nb, bb)[:, :, off:off + 2].copy().view(np.float16).reshape(rows, nb)


def test_q4k_block_fields():
    rng = np.random.default_rng(9)
    rows, cols = 64, 1024
    W = synth.random_q4k_blocks(rng, rows, cols, 1e-2)
    nb = cols // 256
    assert W.shape == (rows, nb * 144)
    for off in (0, 2):                        # d, dmin: finite, >= 0, |N(0, 1e-2)| scale
        v = _fp16_field(W, rows, nb, 144, off).astype(np.float64)
        assert np.isfinite(v).all() and (v >= 0).all()
        assert abs(v.mean() - 1e-2 * np.sqrt(2 / np.pi)) < 1.5e-3
    # code bytes uniform: every 4-bit code about 1/16 of the nibbles
    qs = W.reshape(rows, nb, 144)[:, :, 16:].ravel()
    counts = np.bincount(np.concatenate([qs & 15, qs >> 4]), minlength=16)
    assert (np.abs(counts / counts.sum() - 1 / 16) < 0.01).all()


def test_other_format_scale_fields():
    rng = np.random.default_rng(10)
    rows, cols = 32, 512
    for fmt, offs, signed in ((synth.FMT_Q5_K, (0, 2), False), (synth.FMT_Q6_K, (208,), False),
                              (synth.FMT_Q5_1, (0,), False), (synth.FMT_Q5_1, (2,), True)):
        bw, bb = synth.FMT_BLOCK[fmt]
        nb = cols // bw
        W = synth.random_blocks(rng, fmt, rows, cols, 1e-2)
        assert W.shape == (rows, synth.row_bytes_fmt(fmt, cols)) == (rows, nb * bb)
        for off in offs:
            v = _fp16_field(W, rows, nb, bb, off).astype(np.float64)
            assert np.isfinite(v).all()
            assert ((v < 0).any() if signed else (v >= 0).all()), (fmt, off)


def test_experts_come_from_their_own_streams():
    small = synth.MoE(T=1, E=8, H=256, I=256, top_k=2)
    large = synth.MoE(T=64, E=8, H=256, I=256, top_k=2)
    for e in (0, 5):
        for a, b in zip(small.expert_f32(e), large.expert_f32(e)):
            assert np.array_equal(a, b)
    assert not np.array_equal(small.expert_f32(0)[0], small.expert_f32(1)[0])
    assert small.logits.shape == (1, 8) and large.x.shape == (64, 256)
