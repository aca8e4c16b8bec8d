"""Plant one plausible mistake at a time in a copy of the oracle and require that
some pin catches it.  The planted copies are compiled into a temporary folder on
the CPU; the committed oracle is never modified."""
import os
import subprocess
import sys

import pytest

import oracle
from oracle_pins import PINS

# (name, text in oracle.c, replacement): each a mistake the pages warn about or a
# dropped term, a wrong sign or index, a transposed operand.
MUTANTS = [
    ("exp_instead_of_exp2", "double wa = (a == -INFINITY) ? 0.0 : exp2(a - m);",
     "double wa = (a == -INFINITY) ? 0.0 : exp(a - m);"),
    ("exp_instead_of_exp2_n", "double w = (x == -INFINITY) ? 0.0 : exp2(x - m);",
     "double w = (x == -INFINITY) ? 0.0 : exp(x - m);"),
    ("no_sanitize", "if (isnan(s) || s == INFINITY) return -INFINITY;", ""),
    ("sanitize_nan_only", "if (isnan(s) || s == INFINITY) return -INFINITY;",
     "if (isnan(s)) return -INFINITY;"),
    ("layout_SHN", "double x = sanitize(s[(pos * N + n) * H + h]);",
     "double x = sanitize(s[(pos * H + h) * N + n]);"),
    ("layout_SHN_v", "int64_t off = (pos * N + n) * H + h;", "int64_t off = (pos * H + h) * N + n;"),
    ("range_no_min", "if (end > num_pages) end = num_pages;", ""),
    ("range_floor_pps", "int32_t pps = (num_pages + num_splits - 1) / num_splits;",
     "int32_t pps = num_pages / num_splits;"),
    ("gqa_modulo", "int32_t hk = hq / G;", "int32_t hk = hq % Hkv;"),
    ("natural_log_s", "*s_out = L / log(2.0);", "*s_out = L;"),
    ("dropped_term_b", "if (wb > 0.0) acc += wb * vb[r * D + d];", ""),
    ("merged_s_ln", "s[r] = m + log2(wsum);", "s[r] = m + log(wsum);"),
    ("merged_s_ln_n", "s_out[pos * H + h] = m + log2(wsum);", "s_out[pos * H + h] = m + log(wsum);"),
    ("no_normalise", "v[r * D + d] = acc / wsum;", "v[r * D + d] = acc;"),
    ("no_normalise_n", "for (int64_t d = 0; d < D; ++d) vo[d] = acc[d] / wsum;",
     "for (int64_t d = 0; d < D; ++d) vo[d] = acc[d];"),
    ("slot_index", "return cache + (((pid * Hkv + hk) * page) + (t % page)) * (int64_t)D;",
     "return cache + (((pid * Hkv + hk) * page) + (t / page) % page) * (int64_t)D;"),
    ("no_sm_scale", "score[j] = sm_scale * dot;", "score[j] = dot;"),
    ("sign_flip_max", "double m = a > b ? a : b;", "double m = a < b ? a : b;"),
    ("plan_powers_of_two", "while (ns < 64 && programs * ns < target) ns *= 4;",
     "while (ns < 64 && programs * ns < target) ns *= 2;"),
    ("split_past_ctx", "if (t1 > ctx[b]) t1 = ctx[b];", ""),
    ("no_double_empty_guard",
     "if (a == -INFINITY && b == -INFINITY) {\n            for (int64_t d = 0; d < D; ++d) v[r * D + d] = 0.0;\n            s[r] = -INFINITY;\n            continue;\n        }",
     ""),
    ("cascade_suffix_from_prefix",
     "            for (int32_t t = 0; t < ctx[b]; ++t, ++n) {\n                kr[n] = token_row(k_cache, pages, t, Hkv, hk, page, D);",
     "            for (int32_t t = 0; t < ctx[b]; ++t, ++n) {\n                kr[n] = token_row(k_cache, prefix_pages, t, Hkv, hk, page, D);"),
    ("transposed_v_token", "o[d] += p * vrows[j][d];", "o[d] += p * vrows[n - 1 - j][d];"),
    # multi-level cascade: every level reads level 0's length; the prefix
    # state taken after the suffix; the suffix read from the last shared list
    ("multilevel_level0_length",
     "for (int32_t t = 0; t < seg_len[(int64_t)b * L + l]; ++t, ++n) {",
     "for (int32_t t = 0; t < seg_len[(int64_t)b * L]; ++t, ++n) {"),
    ("multilevel_prefix_state_after_suffix",
     "            attend_rows(D, q + row * D, n, kr, vr, sm_scale, o_pre + row * D, s_pre + row);\n"
     "            for (int32_t t = 0; t < ctx[b]; ++t, ++n) {\n"
     "                kr[n] = token_row(k_cache, sfx, t, Hkv, hk, page, D);\n"
     "                vr[n] = token_row(v_cache, sfx, t, Hkv, hk, page, D);\n"
     "            }\n",
     "            for (int32_t t = 0; t < ctx[b]; ++t, ++n) {\n"
     "                kr[n] = token_row(k_cache, sfx, t, Hkv, hk, page, D);\n"
     "                vr[n] = token_row(v_cache, sfx, t, Hkv, hk, page, D);\n"
     "            }\n"
     "            attend_rows(D, q + row * D, n, kr, vr, sm_scale, o_pre + row * D, s_pre + row);\n"),
    # per-sequence split counts: the largest count used for every sequence;
    # floor instead of ceil; no clamp to the caller's largest count
    ("varlen_uses_max_splits", "oracle_split_range(ctx[b], page, ns, sp, &p0, &p1);",
     "oracle_split_range(ctx[b], page, max_splits, sp, &p0, &p1);"),
    ("plan_varlen_floor", "int32_t ns = (n + pages_per_split - 1) / pages_per_split;",
     "int32_t ns = n / pages_per_split;"),
    ("plan_varlen_no_clamp", "if (ns > max_splits) ns = max_splits;", ""),
    ("multilevel_suffix_from_shared_pages",
     "kr[n] = token_row(k_cache, sfx, t, Hkv, hk, page, D);",
     "kr[n] = token_row(k_cache, seg_pages, t, Hkv, hk, page, D);"),
    ("range_floor_num_pages", "int32_t num_pages = (ctx + page - 1) / page;",
     "int32_t num_pages = ctx / page;"),
    ("merge_states_no_all_empty_guard", "            if (m == -INFINITY) {",
     "            if (0) {"),
    ("empty_split_s_zero", "        *s_out = -INFINITY;", "        *s_out = 0.0;"),
    ("plan_varlen_zero_splits", "if (ns < 1) ns = 1;", ""),
    ("page_index_modulo", "int64_t pid = pages[t / page];", "int64_t pid = pages[t % page];"),
    ("softmax_max_not_subtracted", "z += exp(score[j] - mx);", "z += exp(score[j]);"),
    ("weight_b_from_a", "double wb = (b == -INFINITY) ? 0.0 : exp2(b - m);",
     "double wb = (b == -INFINITY) ? 0.0 : exp2(a - m);"),
    ("cascade_prefix_drops_first_token", "for (int32_t t = 0; t < prefix_len; ++t, ++n) {",
     "for (int32_t t = 1; t < prefix_len; ++t, ++n) {"),
]


_RUNNER = r"""
import sys
sys.path.insert(0, {tests!r})
sys.path.insert(0, {root!r})
import oracle
from oracle_pins import PINS
orc = oracle.Oracle({lib!r})
failed = []
for pin in PINS:
    try:
        pin(orc)
    except Exception as e:
        failed.append(pin.__name__)
print("FAILED_PINS", failed)
sys.exit(1 if failed else 0)
"""


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.SOURCE, encoding="utf-8").read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    path = os.path.join(tmp_path, f"{name}.c")
    with open(path, "w", encoding="utf-8") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_c(path, os.path.join(tmp_path, f"lib{name}.so"))
    tests = os.path.dirname(os.path.abspath(__file__))
    script = _RUNNER.format(tests=tests, root=os.path.dirname(tests), lib=lib)
    # A planted mistake may also crash the process (an index past a buffer):
    # any non-zero exit means the mutant did not survive.
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode != 0, f"no pin caught the planted mistake {name}: {r.stdout}"
