"""The oracle's pins must catch plausible mistakes in the oracle itself.

Each case plants one mistake (a dropped term, a wrong sign or index, a
transposed operand, a missing guard) in a temporary copy of ``kv_oracle.c``,
builds it, and runs the pin suite against that copy: the suite must fail.
Mistakes are planted on the CPU, in the oracle only.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

from oracle.build import SOURCE, build_oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, original text, planted text)
MUTANTS = [
    ("coord_transposed", "return (layer * B + block) * T + token;",
     "return (layer * T + block) * B + token;"),
    ("coord_dropped_layer", "return (layer * B + block) * T + token;",
     "return (block) * T + token;"),
    ("paged_offset_wrong", "    if (b < 0 || b >= B) { *err |= ORC_BAD_BLOCK; return ORC_PAD_SLOT; }\n"
     "    return b * T + p % T;\n}\n\n/* [BT] Datenfluss",
     "    if (b < 0 || b >= B) { *err |= ORC_BAD_BLOCK; return ORC_PAD_SLOT; }\n"
     "    return b * T + (p + 1) % T;\n}\n\n/* [BT] Datenfluss"),
    ("paged_lb_off_by_one", "    int64_t lb = p / T;\n    if (lb >= stride)",
     "    int64_t lb = p / T + 1;\n    if (lb >= stride)"),
    ("paged_null_not_skipped", "    if (b == ORC_NULL_BLOCK) return ORC_PAD_SLOT;\n    if (b < 0 || b >= B) { *err |= ORC_BAD_BLOCK; return ORC_PAD_SLOT; }\n    return b * T + p % T;\n}\n\n/* [BT]",
     "    if (b < 0 || b >= B) { *err |= ORC_BAD_BLOCK; return ORC_PAD_SLOT; }\n    return b * T + p % T;\n}\n\n/* [BT]"),
    ("tail_not_padded",
     "for (int32_t t = 0; t < max_num_tokens; ++t) slot_mapping[t] = ORC_PAD_SLOT;\n"
     "    e |= qsl_errors(qsl, num_reqs, num_tokens);\n    for (int32_t r = 0; r < num_reqs; ++r) {\n"
     "        int32_t lo = qsl[r] < 0 ? 0 : qsl[r];\n"
     "        int32_t hi = qsl[r + 1] > num_tokens ? num_tokens : qsl[r + 1];\n"
     "        const int32_t* row = block_table + (int64_t)r * table_stride;\n"
     "        for (int32_t t = lo; t < hi; ++t)\n"
     "            slot_mapping[t] = paged_slot(",
     "for (int32_t t = 0; t < num_tokens; ++t) slot_mapping[t] = ORC_PAD_SLOT;\n"
     "    e |= qsl_errors(qsl, num_reqs, num_tokens);\n    for (int32_t r = 0; r < num_reqs; ++r) {\n"
     "        int32_t lo = qsl[r] < 0 ? 0 : qsl[r];\n"
     "        int32_t hi = qsl[r + 1] > num_tokens ? num_tokens : qsl[r + 1];\n"
     "        const int32_t* row = block_table + (int64_t)r * table_stride;\n"
     "        for (int32_t t = lo; t < hi; ++t)\n"
     "            slot_mapping[t] = paged_slot("),
    ("range_sign", "int64_t b = (int64_t)rstart[i] + (lb - range_cum);",
     "int64_t b = (int64_t)rstart[i] + (lb + range_cum);"),
    ("range_cum_dropped", "            return b * T + p % T;\n        }\n        range_cum += len;",
     "            return b * T + p % T;\n        }"),
    ("range_bad_len_unflagged", "if (rlen[i] <= 0) return ORC_BAD_RANGE;", "if (rlen[i] < 0) return ORC_BAD_RANGE;"),
    ("write_null_guard_dropped", "if (b == ORC_NULL_BLOCK) { *err |= ORC_NULL_WRITE; return -1; }", ""),
    ("write_src_transposed", "int64_t src = ((int64_t)l * num_tokens + t) * E;",
     "int64_t src = ((int64_t)t * num_layers + l) * E;"),
    ("write_k_v_swapped", "k_cache[n * E + x] = key[src + x];", "k_cache[n * E + x] = value[src + x];"),
    ("gather_offset_dropped",
     "            src_rows[o] = orc_coord(layer, b, p % block_size, num_blocks, block_size);\n"
     "        }\n        o_r += s1 - s0;",
     "            src_rows[o] = orc_coord(layer, b, p % block_size, num_blocks, block_size);\n"
     "        }\n        o_r += 0;"),
    ("gather_range_offset_dropped", "                    break;\n                }\n"
     "                range_cum += len;\n            }\n        }\n        o_r += s1 - s0;",
     "                    break;\n                }\n"
     "                range_cum += len;\n            }\n        }\n        o_r += 0;"),
    ("gather_v_from_k", "v_out[o * E + x] = n >= 0 ? v_cache[n * E + x] : 0;",
     "v_out[o * E + x] = n >= 0 ? k_cache[n * E + x] : 0;"),
    ("gather_token_offset",
     "            src_rows[o] = orc_coord(layer, b, p % block_size, num_blocks, block_size);\n        }",
     "            src_rows[o] = orc_coord(layer, b, (p + 1) % block_size, num_blocks, block_size);\n"
     "        }"),
    ("expand_formula", "out[c * k + j] = (int32_t)(m * k + j);", "out[c * k + j] = (int32_t)(m + j * k);"),
    ("expand_null_expanded", "            if (m == ORC_NULL_BLOCK) continue;\n", ""),
    ("table_from_ranges_offset", "int64_t b = (int64_t)range_start[(int64_t)r * range_stride + i] + j;",
     "int64_t b = (int64_t)range_start[(int64_t)r * range_stride + i] + j + 1;"),
    ("gather_range_sign", "                    int64_t b = (int64_t)rs[i] + (lb - range_cum);",
     "                    int64_t b = (int64_t)rs[i] + (lb + range_cum);"),
    ("gather_range_rows_unvalidated",
     "        e |= range_row_errors(range_len + (int64_t)r * range_stride, num_ranges[r], range_stride);",
     "        (void)0;"),
    ("copy_direction_swapped", "k_cache[d + x] = k_cache[s + x];", "k_cache[s + x] = k_cache[d + x];"),
    ("copy_null_guard_dropped", "if (db == ORC_NULL_BLOCK) { e |= ORC_NULL_WRITE; continue; }", ""),
    ("cp_owner_inverted", "if ((p / I) % W != rank) return ORC_PAD_SLOT;",
     "if ((p / I) % W == rank && W > 1) return ORC_PAD_SLOT;"),
    ("cp_local_offset_dropped_stripe", "return b * T + (v / ((int64_t)I * W)) * I + p % I;",
     "return b * T + (v / I) + p % I;"),
    ("expand_divisor_unchecked", "if (mgr_block_size % kernel_block_size != 0) return ORC_EUNSUPPORTED;", ""),
    ("qsl_order_unchecked", "if (qsl[r] > qsl[r + 1]) e |= ORC_BAD_QSL;", ";"),
    ("qsl_end_unchecked", "if (qsl[0] < 0 || qsl[R] > N) e |= ORC_BAD_QSL;",
     "if (qsl[0] < 0) e |= ORC_BAD_QSL;"),
    ("range_count_unflagged", "if (nr < 0 || nr > range_stride) return ORC_BAD_RANGE;",
     "if (nr < 0 || nr > range_stride) return 0;"),
    ("range_negative_len_counted",
     "        int64_t len = rlen[i] > 0 ? rlen[i] : 0;\n        if (range_cum <= lb",
     "        int64_t len = rlen[i];\n        if (range_cum <= lb"),
    ("range_null_block_written", "            if (b == ORC_NULL_BLOCK) return ORC_PAD_SLOT;\n", ""),
    ("range_malformed_row_resolved", "    if (nr < 0 || nr > range_stride) return ORC_PAD_SLOT;\n",
     "    if (nr < 0) return ORC_PAD_SLOT;\n    if (nr > range_stride) nr = range_stride;\n"),
    ("paged_negative_position_unflagged",
     "if (p < 0) { *err |= ORC_BAD_POSITION; return ORC_PAD_SLOT; }\n    int64_t lb = p / T;\n"
     "    if (lb >= stride)",
     "if (p < 0) { return ORC_PAD_SLOT; }\n    int64_t lb = p / T;\n    if (lb >= stride)"),
    ("write_bad_slot_unflagged", "if (b >= B) { *err |= ORC_BAD_SLOT; return -1; }",
     "if (b >= B) { return -1; }"),
    ("write_v_from_key", "                v_cache[n * E + x] = value[src + x];",
     "                v_cache[n * E + x] = key[src + x];"),
    ("gather_past_row_unflagged",
     "if (lb >= table_stride) { e |= ORC_BAD_POSITION; src_rows[o] = -1; continue; }",
     "if (lb >= table_stride) { src_rows[o] = -1; continue; }"),
    ("gather_bad_span_unflagged",
     "if (s0 < 0 || s1 < s0) { e |= ORC_BAD_POSITION; continue; }\n        const int32_t* row = block_table",
     "if (s0 < 0 || s1 < s0) { continue; }\n        const int32_t* row = block_table"),
    ("gather_out_of_space_unflagged",
     "if (o >= out_rows) { e |= ORC_OUT_OF_SPACE; continue; }\n            int64_t lb = p / block_size;",
     "if (o >= out_rows) { continue; }\n            int64_t lb = p / block_size;"),
    ("gather_range_bad_block_unflagged", "if (b < 0 || b >= num_blocks) e |= ORC_BAD_BLOCK;",
     "if (b < 0 || b >= num_blocks) (void)0;"),
    ("copy_src_null_allowed", "if (sb <= ORC_NULL_BLOCK || sb >= num_blocks)",
     "if (sb < ORC_NULL_BLOCK || sb >= num_blocks)"),
    ("copy_first_layer_only",
     "for (int32_t l = 0; l < num_layers; ++l)\n            for (int32_t t = 0; t < block_size; ++t) {",
     "for (int32_t l = 0; l < 1; ++l)\n            for (int32_t t = 0; t < block_size; ++t) {"),
    ("expand_overflow_unchecked", "if (m < 0 || m * k + (k - 1) > INT32_MAX)", "if (m < 0)"),
    ("table_from_ranges_zero_len_ok", "if (len <= 0) { e |= ORC_BAD_RANGE; continue; }",
     "if (len < 0) { e |= ORC_BAD_RANGE; continue; }"),
    ("table_from_ranges_cut_unflagged", "if (lb >= table_stride) { e |= ORC_OUT_OF_SPACE; break; }",
     "if (lb >= table_stride) { break; }"),
]


def _run_mutant(src, base, mutant):
    """Build one planted copy of the oracle and run the pin suite against it;
    returns the suite's exit code and the end of its output."""
    name, orig, planted = mutant
    if src.count(orig) != 1:
        return None, f"mutation anchor for {name} must occur exactly once"
    d = base / name
    d.mkdir()
    path = d / "kv_oracle_mutant.c"
    path.write_text(src.replace(orig, planted))
    lib = build_oracle(extra_flags=["-Wno-unused-parameter", "-Wno-unused-variable",
                                    "-Wno-unused-but-set-variable"],
                       source=str(path), out=str(d / "libmutant.so"))
    env = dict(os.environ, KV_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    return r.returncode, r.stdout[-2000:]


@pytest.fixture(scope="module")
def mutant_runs(tmp_path_factory):
    """Every planted copy built and pinned, several at a time (each run is its
    own compiler and interpreter process)."""
    src = open(SOURCE).read()
    base = tmp_path_factory.mktemp("mutants")
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        runs = list(ex.map(lambda m: _run_mutant(src, base, m), MUTANTS))
    return {m[0]: r for m, r in zip(MUTANTS, runs)}


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, mutant_runs):
    rc, out = mutant_runs[name]
    assert rc is not None, out
    assert rc != 0, f"planted mistake {name} went unnoticed:\n{out}"
