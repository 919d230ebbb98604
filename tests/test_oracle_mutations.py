"""The pins catch plausible mistakes: each case plants one mistake in a copy of
the oracle's C source (a sign, an index, a dropped term), builds it on the CPU
and runs the pins of that part against it; at least one must fail.  The
oracle itself is not touched."""
import ctypes
import os
import subprocess

import pytest

from oracle import oracle as orc
from tests import test_oracle_formats as fmt_pins
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(orc.__file__), "oracle.c")

MUTATIONS = {
    # Q4_K: the min added instead of subtracted
    "q4k_min_sign": ("out[col] = wq - dm;", "out[col] = wq + dm;",
                     [pins.test_min_is_subtracted, pins.test_hand_built_block_closed_form]),
    # silu on the wrong side of the logistic
    "silu_sign": ("return g / (1.0 + exp(-g));", "return g / (1.0 + exp(g));",
                  [pins.test_silu_closed_forms]),
    # router ties to the higher index
    "router_ties": ("    return ia < ib;\n}", "    return ia > ib;\n}",
                    [pins.test_router_matches_stable_sort_and_softmax,
                     pins.test_router_brute_force_over_all_orders]),
    # RMSNorm without eps under the root
    "rmsnorm_eps": ("double r = 1.0 / sqrt(ss / (double)H + eps);",
                    "double r = 1.0 / sqrt(ss / (double)H);", [pins.test_rmsnorm_worked_example]),
    # Q6_K code offset off by one
    "q6k_offset": ("int q = (lo | (hi << 4)) - 32;", "int q = (lo | (hi << 4)) - 31;",
                   [fmt_pins.test_q6k_closed_form]),
    # Q5_1 offset dropped
    "q51_offset": ("return d * (float)q + m;", "return d * (float)q;",
                   [fmt_pins.test_q51_closed_form_and_partial_rows]),
    # the per-expert down scale divided instead of multiplied
    "moe_scale_div": ("                w *= (double)down_scale[e];", "                w /= (double)down_scale[e];",
                      [pins.test_moe_down_scale_closed_forms]),
    # the per-expert down scale indexed by slot instead of expert
    "moe_scale_slot": ("                w *= (double)down_scale[e];", "                w *= (double)down_scale[j];",
                       [pins.test_moe_down_scale_closed_forms,
                        pins.test_moe_down_scale_recomposed_from_dense_blocks]),
    # Q5_K scale of the wrong sub-block
    "q5k_subblock": ("oracle_q4k_scale_min(scales, k / 32, &sc, &m);\n    int q = q4k_code(qs, k) + 16",
                     "oracle_q4k_scale_min(scales, (k / 32) ^ 1, &sc, &m);\n    int q = q4k_code(qs, k) + 16",
                     [fmt_pins.test_q5k_closed_form]),
}


def build_mutant(tmp_path, name):
    old, new, _ = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                           "-shared", "-o", str(so), str(path), "-lm"])
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    so = build_mutant(tmp_path, name)
    # the wrappers load whatever build() returns: point them at the mutant
    monkeypatch.setattr(orc, "_lib", None)
    monkeypatch.setattr(orc, "build", lambda force=False: so)
    caught = 0
    for test in MUTATIONS[name][2]:
        try:
            test()
        except AssertionError:
            caught += 1
    monkeypatch.setattr(orc, "_lib", None)
    assert caught >= 1, f"no pin caught the mutation {name}"


def test_unmutated_oracle_passes_the_same_pins():
    # (so that the failures above come from the planted mistakes)
    for _, _, tests in MUTATIONS.values():
        for test in tests:
            test()
