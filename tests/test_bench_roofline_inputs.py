"""The algorithmic FLOP and byte counts bench.py divides by (the roofline's
numerators), pinned to the format's arithmetic: Q4_K weights once at 144
bytes per 256 weights (4.5 bits), x once in bf16, y once in fp32, 6*T*H*I
FLOP."""
import bench


def test_dense_layer_counts():
    flop, b = bench.algorithmic("dense", 2048, 4096, 11008, 1, 1)
    assert flop == 6 * 2048 * 4096 * 11008
    wbytes = 2 * 11008 * 16 * 144 + 4096 * 43 * 144
    assert wbytes == 76_087_296                       # 9B-shaped layer, 4.5 bits/weight
    assert b == wbytes + 2048 * 4096 * 2 + 2048 * 4096 * 4 == 126_418_944
    _, b1 = bench.algorithmic("dense", 1, 4096, 11008, 1, 1)
    assert b1 == 76_111_872                           # one decode token
    assert wbytes * 8 / (3 * 4096 * 11008) == 4.5


def test_routed_layer_counts():
    per_expert = 2 * 768 * 8 * 144 + 2048 * 3 * 144
    assert per_expert == 2_654_208
    flop1, b1 = bench.algorithmic("moe", 1, 2048, 768, 128, 8)
    assert flop1 == 6 * 8 * 2048 * 768 and b1 == 8 * per_expert + 2048 * 6
    _, b256 = bench.algorithmic("moe", 256, 2048, 768, 128, 8)
    assert b256 == 128 * per_expert + 256 * 2048 * 6  # every expert touched once
