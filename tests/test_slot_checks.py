"""CPU self-checks of the slot-level GPU checks (slot_cases.py).

1. The constructions hold on the oracle: every dominant slot leads by the
   required margin and the oracle returns its value; a zero query returns the
   plain mean of the attended values, computed here independently.
2. The checks fail on a stand-in for a faulty kernel: copies of the oracle's
   C source with one planted slot mistake (slot 63 of every 64-slot tile left
   out of the softmax; slot 0 of every tile counted twice; the new token
   left out), compiled apart and run in a child process, give outputs that
   the same checks reject.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import workloads as W
from slot_cases import MULTI, SINGLE, UNIT, Step, check_dominant, check_uniform, part_slots, plant_dominant, run_oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")
SRC = os.path.join(ROOT, "oracle", "gqa_oracle.c")

CASES = {c[0]: c for c in SINGLE + UNIT}
MCASES = {c[0]: c for c in MULTI}


def build_step(kind, name, fp8, uniform):
    """The same step the GPU tests build (seeded): returns (step, dominant map)."""
    if kind == "multi":
        _, base, kw, q_lens = MCASES[name]
        st = Step(W.small(base, **kw), "multi", q_lens=q_lens, fp8=fp8)
    else:
        _, base, kw = CASES[name]
        if kind == "attend":
            kw = dict(kw, len_lo=1)
        st = Step(W.small(base, **kw), kind, fp8=fp8)
    dom = None
    if uniform:
        st.t["q"].zero_()
    elif name in dict((c[0], 0) for c in UNIT):
        dom = plant_dominant(st, 15, unit_parts=True)
    else:
        dom = plant_dominant(st, 11, 33 if kind != "multi" else 0)
    st.finish()
    return st, dom


@pytest.mark.parametrize("kind,name,fp8", [("decode", "dense_g4", False), ("decode", "paged16_g6", True),
                                           ("decode", "slots_g8", False), ("attend", "paged16_g6", False),
                                           ("multi", "rows16_g4", False), ("multi", "rows18_g6_paged16", True),
                                           ("multi", "rows32_g4", False), ("multi", "rows40_g8", True),
                                           ("decode", "f32_d64_g4_cap256", False),
                                           ("attend", "slots_g8_cap320", False)])
def test_constructions_hold_on_the_oracle(kind, name, fp8):
    st, dom = build_step(kind, name, fp8, uniform=False)
    out = run_oracle(st)
    assert check_dominant(st, dom, out, out) > 0
    # zero query: the oracle's output is the plain mean of the attended values
    st, _ = build_step(kind, name, fp8, uniform=True)
    out = run_oracle(st)
    for b in range(st.w.B):
        if not st.live(b):
            continue
        for kvh in range(st.w.Hkv):
            _, V = st.unit_kv(b, kvh, st.last[b] + 1)
            for tok, lim in st.rows(b):
                mean = V[:lim + 1].mean(axis=0)
                for h in range(kvh * st.w.G, (kvh + 1) * st.w.G):
                    np.testing.assert_allclose(out[tok, h], mean, rtol=0, atol=1e-12)
    assert check_uniform(st, out, out) == 0.0


MUTANTS = {
    # slot 63 of every 64-slot tile (but the last attended slot) gets no weight
    "tile_slot_dropped": [("    const orc_mods *M = J->mods;\n    if (!M || M->window <= 0)\n        return 1;",
                           "    const orc_mods *M = J->mods;\n    if ((j & 63) == 63 && j < L)\n        return 0;\n"
                           "    if (!M || M->window <= 0)\n        return 1;")],
    # slot 0 of every tile counted twice (numerator and denominator)
    "tile_slot_doubled": [("                Z += exp(s[j] - m);", "                Z += exp(s[j] - m) * (1 + ((j & 63) == 0));"),
                          ("double w = exp(s[j] - m) / Z;", "double w = exp(s[j] - m) * (1 + ((j & 63) == 0)) / Z;")],
    # the new token (slot L) left out of the softmax
    "last_slot_dropped": [("    const orc_mods *M = J->mods;\n    if (!M || M->window <= 0)\n        return 1;",
                           "    const orc_mods *M = J->mods;\n    if (j == L && L > 0)\n        return 0;\n"
                           "    if (!M || M->window <= 0)\n        return 1;")],
}

CHILD = r"""
import sys
import numpy as np
sys.path[:0] = [sys.argv[1], sys.argv[2]]
from test_slot_checks import build_step
from slot_cases import run_oracle
kind, name, fp8, uniform, out = sys.argv[3:]
st, _ = build_step(kind, name, fp8 == "1", uniform == "1")
np.save(out, run_oracle(st))
"""


def _mutant_out(tmp_path, mutant, kind, name, fp8, uniform):
    src = open(SRC).read()
    for before, after in MUTANTS[mutant]:
        assert src.count(before) == 1, f"mutation site for {mutant} not found exactly once"
        src = src.replace(before, after)
    (tmp_path / "m.c").write_text(src)
    lib = tmp_path / "libm.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(lib),
                           str(tmp_path / "m.c"), "-lm"])
    out = tmp_path / "out.npy"
    env = dict(os.environ, GQA_ORACLE_LIB=str(lib))
    subprocess.check_call([sys.executable, "-c", CHILD, ROOT, TESTS, kind, name, "1" if fp8 else "0",
                           "1" if uniform else "0", str(out)], env=env, timeout=600)
    return np.load(out)


@pytest.mark.parametrize("kind,name,fp8", [("decode", "dense_g4", False), ("multi", "rows16_g4", True)])
@pytest.mark.parametrize("mutant", ["tile_slot_dropped", "last_slot_dropped"])
def test_dominant_check_rejects_a_lost_slot(tmp_path, mutant, kind, name, fp8):
    got = _mutant_out(tmp_path, mutant, kind, name, fp8, uniform=False)
    st, dom = build_step(kind, name, fp8, uniform=False)
    want = run_oracle(st)
    with pytest.raises(AssertionError):
        check_dominant(st, dom, got, want)


@pytest.mark.parametrize("kind,name,fp8", [("decode", "paged16_g6", False), ("multi", "rows8_g4", False)])
@pytest.mark.parametrize("mutant", ["tile_slot_dropped", "tile_slot_doubled", "last_slot_dropped"])
def test_zero_query_check_rejects_a_wrong_slot_count(tmp_path, mutant, kind, name, fp8):
    got = _mutant_out(tmp_path, mutant, kind, name, fp8, uniform=True)
    st, _ = build_step(kind, name, fp8, uniform=True)
    want = run_oracle(st)
    with pytest.raises(AssertionError):
        check_uniform(st, got, want)


def test_unit_part_edges_are_planted():
    """The small-cache construction puts j* on a part edge of a 2-, 4- or
    8-CTA cluster in every unit whose row has such an edge."""
    _, base, kw = CASES["f32_d64_g4_cap256"]
    st = Step(W.small(base, **kw), "decode")
    dom = plant_dominant(st, 15, unit_parts=True)
    k = 0
    for b in range(st.w.B):
        if not st.live(b):
            continue
        for kvh in range(st.w.Hkv):
            edges = part_slots(st, b, k)
            if edges:
                assert dom[(b, kvh)] in edges
            k += 1
