"""The pins must catch plausible mistakes in the oracle.

Each case copies the oracle's C source, plants one mistake (a dropped term, a
wrong index or sign, a transposed operand, a skipped step), compiles the copy
into a temporary directory and runs the pin tests against it in a child
process. The pins pass on the real oracle and must fail on every mutant.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gqa_oracle.c")

MUTANTS = {
    "strided_groups": ("const int h = kvh * G + g;", "const int h = g * J->Hkv + kvh;"),
    "no_scale": ("s[j] = dot / sqrt((double)D);", "s[j] = dot;"),
    "scale_by_d": ("s[j] = dot / sqrt((double)D);", "s[j] = dot / (double)D;"),
    "new_token_dropped": ("        for (int j = 0; j <= L; ++j) {\n            double dot",
                          "        for (int j = 0; j < L; ++j) {\n            double dot"),
    "stale_slot_counted": ("        for (int j = 0; j <= L; ++j)\n            if (attended(J, b, L, j))\n                Z += exp(s[j] - m);",
                           "        for (int j = 0; j <= L + 1 && j < 2 * L + 1; ++j)\n            if (attended(J, b, L, j < L + 1 ? j : L))\n                Z += exp(s[j < L + 1 ? j : L] - m);"),
    "window_off_by_one": ("if (j > L - M->window)", "if (j >= L - M->window)"),
    "prefix_inclusive": ("    return j < P;\n}", "    return j <= P;\n}"),
    "sink_scaled": ("double Z = sink ? exp((double)sink[h] - m) : 0.0;",
                    "double Z = sink ? exp((double)sink[h] / sqrt((double)D) - m) : 0.0;"),
    "sink_dropped": ("double Z = sink ? exp((double)sink[h] - m) : 0.0;", "double Z = 0.0;"),
    "prefix_rows_ignored": ("const int P = M->kept_prefix_rows ? M->kept_prefix_rows[b] : M->kept_prefix;",
                            "const int P = M->kept_prefix;"),
    "masked_slot_weighted": ("            if (!attended(J, b, L, j))\n                continue;\n", ""),
    "sign_flip": ("                Z += exp(s[j] - m);", "                Z += exp(m - s[j]);"),
    "row_head_swapped": ("return ((r * lay->Hkv + kvh) * lay->Smax + s) * lay->D;",
                         "return ((kvh * lay->Hkv + r % lay->Hkv) * lay->Smax + s) * lay->D;"),
    "paged_offset": ("(size_t)(s % lay->block_size)) * lay->D;", "(size_t)(s / lay->block_size)) * lay->D;"),
    "append_skipped": ("    if (!J->attend && J->do_append) {\n        size_t dst", "    if (0) {\n        size_t dst"),
    "slot_ids_ignored": ("size_t r = lay->slot_ids ? (size_t)lay->slot_ids[b] : (size_t)b;", "size_t r = (size_t)b;"),
    "duplicates_accepted": ("if (slot_ids[c] == slot_ids[b])", "if (0)"),
    "paged_repeat_accepted": ("if (row[k] == row[i])", "if (0)"),
    "bf16_shift": ("[i] << 16;", "[i] << 15;"),
    "attend_stale_slot": ("const int L = J->attend ? J->lengths[b] - 1 : J->lengths[b];",
                          "const int L = J->lengths[b];"),
    "attend_query_rounded": ("dot += elem(J->q, q_i + d, J->q_dtype) * kd;",
                             "{ double x = elem(J->q, q_i + d, J->q_dtype);"
                             " if (x != 0) x = ldexp(nearbyint(ldexp(x, 7 - ilogb(x))), ilogb(x) - 7);"
                             " dot += x * kd; }"),
    "attend_empty_accepted": ("if (last_slot(lengths, b, attend) < 0 ||", "if (last_slot(lengths, b, attend) < -1 ||"),
    "paged_last_block_unchecked": ("for (long long i = 0; i <= last / block_size; ++i)",
                                   "for (long long i = 0; i < last / block_size; ++i)"),
    "multi_not_causal": ("attend_heads(J, b, kvh, Lb + i, t0 + i, J->do_append ? INT_MAX : Lb, t0);",
                         "attend_heads(J, b, kvh, Lb + nq - 1, t0 + i, J->do_append ? INT_MAX : Lb, t0);"),
    "multi_append_offset": ("size_t dst = slot_index(&J->lay, b, kvh, Lb + i);",
                            "size_t dst = slot_index(&J->lay, b, kvh, Lb + i + (i > 0));"),
    "multi_same_token_appended": ("append_vec(J, J->k_cache, dst, J->k_new, new_index(J, t0 + i, kvh), KS, kvh);",
                                  "append_vec(J, J->k_cache, dst, J->k_new, new_index(J, t0, kvh), KS, kvh);"),
    "multi_cu_q_unchecked": ("        if (cu_q[b + 1] < cu_q[b])\n            return ORC_INVALID_ARGUMENT;\n", ""),
    "e4m3_exponent_bias": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    "e4m3_ties_away": ("(lo & 1) ? hi : lo", "hi"),
    "e4m3_scale_not_applied": ("return (double)scale[kvh] * orc_e4m3_decode(((const uint8_t *)cache)[i]);",
                               "return orc_e4m3_decode(((const uint8_t *)cache)[i]);"),
    "e4m3_append_not_divided": ("const float y = (float)elem(news, src + d, J->new_dtype) / scale[kvh];",
                                "const float y = (float)elem(news, src + d, J->new_dtype);"),
    "e4m3_new_unquantised": ("    if (J->kv_dtype != ORC_E4M3)\n        return x;\n    const float y = (float)x / scale[kvh];",
                             "    if (1)\n        return x;\n    const float y = (float)x / scale[kvh];"),
    "query_head_offset": ("const size_t q_i = ((size_t)tok * J->Hq + h) * D;", "const size_t q_i = ((size_t)tok * J->Hq + g) * D;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation site for {name} not found exactly once"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(before, after))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-o", str(lib), str(mut), "-lm"])
    env = dict(os.environ, GQA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
