"""The pins are strong enough: each plausible mistake planted in a copy of the
oracle source (a dropped term, a wrong sign, index, shift or operand) must make
at least one pin in test_oracle_pins.py fail.  Mistakes are planted only in
temporary copies of the C source, compiled and loaded on the CPU."""
import os
import subprocess
import tempfile

import pytest

import oracle
import tests.test_oracle_pins as pins

Q4_K, Q5_K, Q6_K = 1, 2, 3

# (name, original text, mutated text)
MUTANTS = [
    ("drop min term", "- dmin * (double)f.m[j]", ""),
    ("q6 zero point", "(double)(f.q[i] - 32)", "(double)(f.q[i] - 31)"),
    ("q6 scale index", "f.sc[i / 16]", "f.sc[i / 32]"),
    ("q4 sub-block index", "int j = i / 32;", "int j = (i / 16) % 8;"),
    ("scale high bits from wrong byte", "((s[j - 4] >> 6) << 4)", "((s[j] >> 6) << 4)"),
    ("min high bits from wrong byte", "((s[j] >> 6) << 4);\n    }\n}", "((s[j - 4] >> 6) << 4);\n    }\n}"),
    ("nibbles swapped", "f->q[64 * g + l] = lo;\n                f->q[64 * g + 32 + l] = hi;",
     "f->q[64 * g + l] = hi;\n                f->q[64 * g + 32 + l] = lo;"),
    ("q5 fifth bit position", "lo |= ((qh[l] >> (2 * g)) & 1) << 4;", "lo |= ((qh[l] >> g) & 1) << 4;"),
    ("q6 high bit pair", "(b & 15) | (((c >> 2) & 3) << 4)", "(b & 15) | (((c >> 4) & 3) << 4)"),
    ("q6 low nibble source", "f->q[128 * h + 64 + l] = (a >> 4)", "f->q[128 * h + 64 + l] = (b >> 4)"),
    ("fp16 exponent bias", "ldexp(1024.0 + (double)f, e - 25)", "ldexp(1024.0 + (double)f, e - 24)"),
    ("fp16 subnormal scale", "ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    ("x reversed", "x_value(x, x_dtype, x_off + k)", "x_value(x, x_dtype, x_off + (K - 1 - k))"),
    ("last weight dropped", "if (k >= K) break;", "if (k >= K - 1) break;"),
    ("abs sum signed", "acc_abs += fabs(t);", "acc_abs += t;"),
    ("gate dropped", "acc += g * p[(m * top_k + t) * N + n];", "acc += p[(m * top_k + t) * N + n];"),
    ("dmin read from d", "f->dmin_bits = rd16(blk + 2);", "f->dmin_bits = rd16(blk);"),
    ("ia4 bias dropped", "scale * (double)(byte & 15) + bias;", "scale * (double)(byte & 15);"),
    ("ia4 nibbles swapped", "w[64 * g + 32 + l] = scale * (double)(byte >> 4) + bias;",
     "w[64 * g + 32 + l] = scale * (double)(byte & 15) + bias;"),
    ("ia4 bias read from the scales", "oracle_bf16_to_double(rd16(blk + 8 + 2 * g))",
     "oracle_bf16_to_double(rd16(blk + 2 * g))"),
    ("ia4 group index", "double scale = oracle_bf16_to_double(rd16(blk + 2 * g));",
     "double scale = oracle_bf16_to_double(rd16(blk + 2 * (g & 1)));"),
]

# every pin, with one set of arguments each
CHECKS = (
    [(pins.test_block_sizes, {}), (pins.test_half_decoder_all_patterns, {}),
     (pins.test_golden_handbuilt_blocks, {}), (pins.test_q6k_zero_point_and_one_hot, {}),
     (pins.test_moe_rejects_bad_expert_id, {})]
    + [(pins.test_moe_matches_per_slot_products, {"with_gate": wg, "x_per_slot": xs})
       for wg in (False, True) for xs in (False, True)]
    + [(f, {"qtype": t}) for t in (Q4_K, Q5_K) for f in
       (pins.test_closed_form_constant_fields, pins.test_one_hot_scale_and_min)]
    + [(f, {"qtype": t}) for t in (Q4_K, Q5_K, Q6_K) for f in
       (pins.test_dequant_matches_bit_reader_and_rounds_once, pins.test_matvec_linearity_and_zero,
        pins.test_matvec_weights_past_K_ignored)]
    + [(pins.test_matvec_brute_force, {"qtype": t, "NK": (3, 512)}) for t in (Q4_K, Q5_K, Q6_K)]
    + [(pins.test_matvec_integer_special_case, {"qtype": t, "x_dtype": "f32"}) for t in (Q4_K, Q5_K, Q6_K)]
    + [(pins.test_unpack_matches_bit_reader, {"qtype": t}) for t in (Q4_K, Q5_K, Q6_K)]
    + [(pins.test_ia4_pack_then_block_decode_equals_mlx_definition, {}), (pins.test_ia4_hand_worked_block, {}),
       (pins.test_ia4_matvec_reduces_to_dense_integer_product, {})]
)


def _any_pin_fails() -> bool:
    for fn, kw in CHECKS:
        try:
            fn(oracle, **kw)
        except (AssertionError, ValueError):
            return True
    return False


def test_unmutated_oracle_passes_every_check():
    oracle.use_library(None)
    assert not _any_pin_fails()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {name}"
    with tempfile.TemporaryDirectory() as tmp:
        csrc = os.path.join(tmp, "kq_oracle.c")
        with open(csrc, "w") as fh:
            fh.write(src.replace(old, new))
        with open(os.path.join(tmp, "kq_oracle.h"), "w") as fh:
            fh.write(open(os.path.join(oracle.HERE, "kq_oracle.h")).read())
        so = os.path.join(tmp, "libmutant.so")
        subprocess.check_call(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-o", so, csrc, "-lm"])
        oracle.use_library(so)
        try:
            assert _any_pin_fails(), f"planted mistake not caught: {name}"
        finally:
            oracle.use_library(None)
