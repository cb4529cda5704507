"""The pins catch plausible mistakes: each case plants one mistake in a copy of
the oracle (on the CPU, in a temporary directory), loads that copy in place of
the real one, and checks that at least one pin of test_oracle_pins fails."""
from __future__ import annotations

import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, original text, planted text); each original must occur in oracle.c
MUTANTS = [
    ("dropped_last_rank", "for (int p = 1; p < n; ++p)\n        acc = acc + orc_bf16_to_f32(x[p][i]);\n    return orc_f32_to_bf16(acc);\n}\n\nuint16_t orc_fold_zero_start",
     "for (int p = 1; p < n - 1; ++p)\n        acc = acc + orc_bf16_to_f32(x[p][i]);\n    return orc_f32_to_bf16(acc);\n}\n\nuint16_t orc_fold_zero_start"),
    ("wrong_sign", "acc = acc + orc_bf16_to_f32(x[p][i]);\n    return orc_f32_to_bf16(acc);\n}\n\nuint16_t orc_fold_zero_start",
     "acc = acc - orc_bf16_to_f32(x[p][i]);\n    return orc_f32_to_bf16(acc);\n}\n\nuint16_t orc_fold_zero_start"),
    ("reversed_rank_order", "float acc = orc_bf16_to_f32(x[0][i]);\n    for (int p = 1; p < n; ++p)\n        acc = acc + orc_bf16_to_f32(x[p][i]);",
     "float acc = orc_bf16_to_f32(x[n - 1][i]);\n    for (int p = n - 2; p >= 0; --p)\n        acc = acc + orc_bf16_to_f32(x[p][i]);"),
    ("ties_away_from_zero", "dropped > 0x8000u ||", "dropped >= 0x8000u ||"),
    ("truncation", "kept += 1u;", "kept += 0u;"),
    ("nan_not_canonical", "return (uint16_t)0x7FC0u;", "return (uint16_t)(u >> 16);"),
    ("widening_shift", "(uint32_t)b << 16;", "(uint32_t)b << 15;"),
    ("shard_not_rounded", "return (per + 7u) / 8u * 8u;", "return per;"),
    ("rs_wrong_index", "out[r][j] = orc_fold(in, n, b + j);", "out[r][j] = orc_fold(in, n, j);"),
    ("a2a_transposed", "in[p][(size_t)d * m + j]", "in[d][(size_t)p * m + j]"),
    ("ag_wrong_slot", "out[d][b + j] = in[p][j];", "out[d][j] = in[p][j];"),
    ("ll8_swapped_halves", "lines[j] = lo | (hi << 16) | (flag << 32);", "lines[j] = hi | (lo << 16) | (flag << 32);"),
    ("ll8_decode_ignores_flag", "if ((uint32_t)(line >> 32) != (uint32_t)epoch) {", "if (0) {"),
    ("ll128_big_endian_seq", "line[120 + b] = (uint8_t)((epoch >> (8 * b)) & 0xFFu);", "line[120 + b] = (uint8_t)((epoch >> (8 * (7 - b))) & 0xFFu);"),
    ("ll128_59_per_line", "size_t idx = j * 60u + q;\n            uint16_t v", "size_t idx = j * 59u + q;\n            uint16_t v"),
    ("moe_source_transposed", "counts[e * n + p] += 1;", "counts[e * n + (n - 1 - p)] += 1;"),
    ("rsv_offset_not_advanced", "            out[r][j] = orc_fold(in, n, off + j);\n        off += len[r];", "            out[r][j] = orc_fold(in, n, off + j);\n        off += 0;"),
    ("a2av_source_offset", "                src += len[(size_t)p * n + k];", "                src += len[(size_t)k * n + p];"),
    ("agv_rank_order", "                out[d][off + j] = in[p][j];\n            off += len[p];", "                out[d][off + j] = in[n - 1 - p][j];\n            off += len[p];"),
    ("sent_sanitizes_wrong_pattern", "if (x == ORC_SENT_BF16)", "if (x == 0x7FFFu)"),
    ("sent_packs_big_endian", "pack |= v << (16 * q);", "pack |= v << (16 * (3 - q));"),
    ("sent_decode_accepts_sentinel", "if (pack == ~(uint64_t)0) {", "if (0) {"),
    ("sent_not_sanitized_in_encode", "uint64_t v = idx < elems ? orc_sent_sanitize(in[idx]) : 0u;",
     "uint64_t v = idx < elems ? in[idx] : 0u;"),
    ("f32_nan_keeps_payload", "        return 0x7FC00000u; /* any NaN: the canonical quiet NaN */",
     "        memcpy(&u, &f, sizeof u); return u;"),
    ("f32_fold_drops_rank0", "    float acc = f32_of(x[0][i]);\n    for (int p = 1; p < n; ++p)\n        acc = acc + f32_of(x[p][i]);",
     "    float acc = 0.0f;\n    for (int p = 1; p < n; ++p)\n        acc = acc + f32_of(x[p][i]);"),
    ("f32_rs_wrong_offset", "            out[r][j] = orc_fold_f32(in, n, b + j);", "            out[r][j] = orc_fold_f32(in, n, j);"),
    ("f32_sent_pack_swapped", "        packs[j] = lo | (hi << 32);", "        packs[j] = hi | (lo << 32);"),
    ("f32_sent_decode_accepts_sentinel", "        if (pack == 0xFFFFFFFFFFFFFFFFull) { /* not yet published */", "        if (0) {"),
    ("f32_sent_wrong_pattern", "    if (x == 0xFFFFFFFFu)\n        return 0x7FC00000u;", "    if (x == 0xFFFF0000u)\n        return 0x7FC00000u;"),
    ("copy_drops_first_byte", "    for (size_t i = 0; i < bytes; ++i)\n        dst[i] = src[i];",
     "    for (size_t i = 1; i < bytes; ++i)\n        dst[i] = src[i];"),
    ("copy_reversed", "        dst[i] = src[i];", "        dst[i] = src[bytes - 1 - i];"),
    ("moe_source_major_order", "for (int le = 0; le < el; ++le) {\n            int e = d * el + le;\n            for (int p = 0; p < n; ++p)",
     "for (int le = 0; le < el; ++le) {\n            int e = d * el + le;\n            for (int p = n - 1; p >= 0; --p)"),
]

# Pins that need only the `orc` handle (the exhaustive rounding sweep and the
# torch cross-checks are left out: they are slow and the hand cases and the
# exact-rational brute force already cover rounding).
PINS = [
    pins.test_rounding_hand_cases,
    pins.test_widening_all_patterns_match_field_decoding,
    lambda o: pins.test_fold_integer_inputs_sum_exactly(o, 8),
    pins.test_fold_n1_is_identity_for_every_non_nan_pattern,
    pins.test_fold_rank_order_is_observable,
    pins.test_fold_bruteforce_n3_to_n8_against_exact_rationals,
    pins.test_fold_overflow_and_subnormals,
    pins.test_figure4_worked_example,
    lambda o: pins.test_allreduce_invariants(o, 3, 1000),
    pins.test_shard_geometry_closed_forms,
    pins.test_all_to_all_is_an_involution_and_a_permutation,
    pins.test_all_gather_is_rank_ordered_concatenation,
    pins.test_ll8_line_layout_hand_case,
    pins.test_ll8_rejects_any_other_flag,
    pins.test_ll128_line_layout_hand_case,
    pins.test_ll128_rejects_other_sequence_numbers,
    pins.test_moe_tiny_hand_derived_layout,
    pins.test_v_collectives_invariants_on_zipf_splits,
    pins.test_all_to_all_v_hand_case,
    pins.test_moe_counts_and_rows_invariants,
    pins.test_sentinel_sanitize_changes_only_the_reserved_nan,
    pins.test_sentinel_pack_layout_hand_case,
    pins.test_sentinel_roundtrip_every_pattern_in_every_position,
    pins.test_sentinel_pack_is_not_ready,
    pins.test_fold_f32_special_values,
    pins.test_fold_f32_n1_is_identity,
    pins.test_reduce_scatter_f32_is_the_allreduce_partition,
    pins.test_sentinel_f32_sanitize_and_layout,
    pins.test_one_sided_copy_delivers_every_byte_in_order,
]


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, orig, planted, tmp_path, monkeypatch):
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert src.count(orig) == 1, f"mutation anchor for {name} not unique"
    mdir = tmp_path / "m"
    mdir.mkdir()
    (mdir / "oracle.c").write_text(src.replace(orig, planted))
    (mdir / "oracle.h").write_text(open(os.path.join(ROOT, "oracle", "oracle.h")).read())
    so = str(mdir / "liboracle_mutant.so")
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-o", so, str(mdir / "oracle.c")])
    mutant = ctypes.CDLL(so)
    oracle._declare(mutant)
    monkeypatch.setattr(oracle, "_lib", mutant)
    caught = []
    for pin in PINS:
        try:
            pin(oracle)
        except (AssertionError, ValueError) as exc:  # a pin rejected the mutant
            caught.append((getattr(pin, "__name__", "pin"), type(exc).__name__))
            break
    assert caught, f"no pin catches the planted mistake {name}"
