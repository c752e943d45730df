"""Planted mistakes in the oracle must be caught by the pins.

Each mutant is a copy of oracle/tide_oracle.c with one plausible mistake (a
dropped term, a wrong sign, a wrong index or offset, a reversed order, a
wrong zero) compiled into a temporary library.  The pins of oracle_pins.py
run against it in a child process (so a mutant that crashes cannot take the
test run down); at least one of them must fail.  The mistakes are planted in
the oracle on the CPU only.
"""
import os
import subprocess
import sys
import textwrap

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

MUTANTS = {
    "drop_rank1_term": [("for (int32_t u = 1; u < world; ++u)\n            acc = acc +",
                         "for (int32_t u = 2; u < world; ++u)\n            acc = acc +")],
    "wrong_sign": [("acc = acc + pack[", "acc = acc - pack[")],
    "reversed_order": [("float acc = pack[j];", "float acc = pack[(size_t)(world - 1) * (size_t)n + (size_t)j];"),
                       ("acc = acc + pack[(size_t)u * (size_t)n", "acc = acc + pack[(size_t)(world - 1 - u) * (size_t)n")],
    "seed_from_plus_zero": [("float acc = pack[j];", "float acc = 0.0f + pack[j];")],
    "negative_zero_padding": [("dst[j] = 0.0f;", "dst[j] = -0.0f;")],
    "floor_rows": [("int64_t R = (dim0[p] + world - 1) / world;", "int64_t R = dim0[p] / world + 1;")],
    "source_row_offset": [("src[u] = grads[(size_t)p * (size_t)world + (size_t)u] + (size_t)r * (size_t)R[p] * (size_t)K;",
                           "src[u] = grads[(size_t)p * (size_t)world + (size_t)u] + (size_t)r * (size_t)K;")],
    "unscaled_accumulate": [("out[j] = accumulate ? old[j] + y : y;", "out[j] = accumulate ? old[j] + acc : y;")],
    "scale_before_sum": [("float y = alpha * acc;", "float y = acc;"),
                         ("dst[j] = bf16_to_f32(src[u][j]);", "dst[j] = alpha * bf16_to_f32(src[u][j]);")],
    "ag_drops_offset": [("const uint16_t *from = slots + (size_t)r * (size_t)stride + (size_t)o[p] +",
                         "const uint16_t *from = slots + (size_t)r * (size_t)stride +")],
    "ag_transposed_rank": [("uint16_t *to = full[p] + (size_t)((r * R[p] + i) * K);",
                            "uint16_t *to = full[p] + (size_t)((i * (int64_t)world + r) * K);")],
    "offset_without_padding": [("off += R * row_numel[p];", "off += (dim0[p] * row_numel[p] + world - 1) / world;")],
    "cast_truncates": [("if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))", "if (0)")],
    "cast_ties_away": [("(dropped == 0x8000u && (kept & 1u))", "(dropped == 0x8000u)")],
    "cast_drops_nan": [("        return (uint16_t)((w >> 16) | 0x0040u);", "        return (uint16_t)0x7F80u;")],
    "ag_cast_drops_offset": [("const float *src_row = slots + (size_t)r * (size_t)stride + (size_t)o[p] +",
                              "const float *src_row = slots + (size_t)r * (size_t)stride +")],
    "ex_negative_zero_padding": [("            dst[j] = +0.0f;", "            dst[j] = -0.0f;")],
    "ex_unscaled_accumulate": [("out[j] = accumulate ? (old[j] + y) : y;", "out[j] = accumulate ? (old[j] + total) : y;")],
    "ex_last_partial_dropped": [("for (int32_t g0 = 0; g0 < world; g0 += group) {",
                                 "for (int32_t g0 = 0; g0 + group < world || g0 == 0; g0 += group) {")],
    "staged_own_first": [("        seq[q] = r;\n", "        seq[q] = seq[0];\n        seq[0] = r;\n")],
    "nodes_owner_fixed": [("int32_t owner = n * node_size + r % node_size;", "int32_t owner = n * node_size;")],
    "nodes_as_one_chain": [("        *group = node_size;", "        *group = world;")],
    "f32_grads_truncated": [("    return ((const float *)src)[j];",
                             "    return bf16_to_f32((uint16_t)(((const uint32_t *)src)[j] >> 16));")],
    "tree_as_rank_order": [("        if (order == ORACLE_ORDER_TREE) {", "        if (0) {")],
    "tree_far_pairs": [("level[i] = level[2 * i] + level[2 * i + 1];", "level[i] = level[i] + level[i + m / 2];")],
    "tree_odd_value_dropped": [("                    level[m / 2] = level[m - 1];", "                    ;")],
    "ag_cast_transposed_rank": [("uint16_t *dst_row = full[p] + (size_t)((r * R[p] + i) * K);",
                                 "uint16_t *dst_row = full[p] + (size_t)((i * (int64_t)world + r) * K);")],
}

RUNNER = textwrap.dedent("""
    import sys
    sys.path[:0] = [{root!r}, {tests!r}]
    import oracle
    from oracle_pins import ALL_PINS
    orc = oracle.Oracle({lib!r})
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError as e:
            caught.append(pin.__name__)
        except (ValueError, MemoryError) as e:
            caught.append(pin.__name__ + ':' + type(e).__name__)
    print('CAUGHT', ' '.join(caught))
""")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    with open(oracle.SOURCE) as f:
        src = f.read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
        src = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(src)
    lib = oracle.compile_library(str(path), str(tmp_path / "libmutant.so"))
    code = RUNNER.format(root=ROOT, tests=HERE, lib=lib)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    caught = [l for l in res.stdout.splitlines() if l.startswith("CAUGHT")]
    if res.returncode != 0 and not caught:
        return  # the mutant crashed the checker outright: caught
    assert caught, res.stdout + res.stderr
    assert caught[0].split()[1:], f"mutant {name} passed every pin"
