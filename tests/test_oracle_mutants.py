"""The pins must catch plausible mistakes in the oracle.

Each case copies ddp_oracle.c into a temporary directory, plants one
plausible mistake in the copy (wrong chunk index, wrong neighbour, dropped
divide, wrong rounding, wrong cap comparison, ...), builds it and runs the
oracle pin tests against it (the loader honours DDP_ORACLE_LIB).  Every
mutant must fail at least one pin.  The committed oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ddp_oracle.c")
PINS = ["tests/test_oracle_ring.py", "tests/test_oracle_plan.py", "tests/test_oracle_tree.py",
        "tests/test_oracle_fp16.py"]

MUTANTS = {
    "rs_send_chunk_off_by_one": ("? mod((int64_t)r - s, world) :", "? mod((int64_t)r - s - 1, world) :"),
    "ag_send_chunk_off_by_one": (": mod((int64_t)r - s + 1, world);", ": mod((int64_t)r - s, world);"),
    "receive_from_right_neighbour": ("int32_t left = mod((int64_t)r - 1, world);",
                                     "int32_t left = mod((int64_t)r + 1, world);"),
    "divide_dropped": ("if (n_steps < 0 && divisor > 1)", "if (0)"),
    "divide_by_reciprocal": ("p[i] = p[i] / dv;", "p[i] = p[i] * (1.0f / dv);"),
    "overwrite_instead_of_add": ("d[i] = d[i] + s[i];", "d[i] = s[i];"),
    "subtract_instead_of_add": ("d[i] = d[i] + s[i];", "d[i] = d[i] - s[i];"),
    "floor_chunk_size": ("return N > 0 ? (S + N - 1) / N : 0;", "return N > 0 ? S / N : 0;"),
    "bf16_ties_away": ("(dropped == 0x8000u && (kept & 1u))", "(dropped == 0x8000u)"),
    "bf16_truncate_per_hop": (
        "d[i] = oracle_bf16_rne(oracle_bf16_to_f32(d[i]) + oracle_bf16_to_f32(s[i]));",
        "d[i] = (uint16_t)(f32_bits(oracle_bf16_to_f32(d[i]) + oracle_bf16_to_f32(s[i])) >> 16);"),
    "plan_strict_cap": ("if (elems * elem_bytes >= cap) {", "if (elems * elem_bytes > cap) {"),
    "plan_forward_order": ("for (int32_t p = n_params - 1; p >= 0; --p) {",
                           "for (int32_t p = 0; p < n_params; ++p) {"),
    "plan_first_cap_everywhere": ("int64_t cap = (k == 0) ? first_cap_bytes : cap_bytes;",
                                  "int64_t cap = first_cap_bytes;"),
    "tree_reduce_distances_reversed": ("const int32_t d = reduce ? (1 << step) : (1 << (total_steps - 1 - step));",
                                       "const int32_t d = reduce ? (1 << (depth - 1 - step)) : (1 << (total_steps - 1 - step));"),
    "tree_broadcast_wrong_sender": ("if (r % (2 * d) == d) memcpy(bufs[r], msg[r - d], bytes);",
                                    "if (r % (2 * d) == d) memcpy(bufs[r], msg[r], bytes);"),
    "tree_divide_dropped": ("if (n_steps < 0 && reduce && step == depth - 1 && divisor > 1)", "if (0)"),
    "plan_drops_trailing_bucket": ("    if (members > 0) {\n        bucket_numel[k] = elems;",
                                   "    if (0) {\n        bucket_numel[k] = elems;"),
    "pack_offset_in_elements_not_bytes": (
        "memcpy((char*)bucket + offset[i] * elem_bytes, grads[i], (size_t)(numel[i] * elem_bytes));",
        "memcpy((char*)bucket + offset[i], grads[i], (size_t)(numel[i] * elem_bytes));"),
    "unpack_short_by_one_element": (
        "memcpy(grads[i], (const char*)bucket + offset[i] * elem_bytes, (size_t)(numel[i] * elem_bytes));",
        "memcpy(grads[i], (const char*)bucket + offset[i] * elem_bytes, (size_t)((numel[i] - 1) * elem_bytes));"),
    "accumulate_skipped": ("    if (n > 0) add_into(dtype, acc, g, n);", "    (void)acc; (void)g;"),
    "fp16_ties_away": ("if (rem > half || (rem == half && (kept & 1u))) kept += 1u;",
                       "if (rem >= half) kept += 1u;"),
    "fp16_subnormals_flushed": ("    if (shift > 40) return sign;", "    if (E < -14) return sign;"),
    "fp16_overflow_saturates": ("        if (be >= 31) return (uint16_t)(sign | 0x7C00u);",
                                "        if (be >= 31) return (uint16_t)(sign | 0x7BFFu);"),
    "bf16_divide_rounds_toward_zero": (
        "for (int64_t i = 0; i < n; ++i) p[i] = oracle_bf16_rne(oracle_bf16_to_f32(p[i]) / dv);",
        "for (int64_t i = 0; i < n; ++i) p[i] = (uint16_t)(f32_bits(oracle_bf16_to_f32(p[i]) / dv) >> 16);"),
}


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut = tmp_path / "ddp_oracle_mutant.c"
    mut.write_text(src.replace(old, new), encoding="utf-8")
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                           "-o", str(so), str(mut)])
    env = dict(os.environ, DDP_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
