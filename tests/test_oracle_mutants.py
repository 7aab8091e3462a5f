"""Planted mistakes in the oracle must trip its pins (CPU only).

Each case copies ``oracle/nf4_oracle.c``, applies one textual change that a plausible slip would
make, builds the copy into a temporary library and runs the fast pins of ``oracle_pins.py``
against it.  At least one pin must fail; otherwise the pins would let that mistake through.
"""
import os

import pytest

import oracle
import oracle_pins as P

MUTANTS = [
    ("nibble order swapped",
     "codes[j] = (uint8_t)(lo | (hi << 4));", "codes[j] = (uint8_t)(hi | (lo << 4));"),
    ("unpacking reads the high nibble first",
     "return (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);", "return (k % 2 == 1) ? (byte & 0x0F) : (byte >> 4);"),
    ("ties go to the higher index", "if (d < best_d) {", "if (d <= best_d) {"),
    ("scale stored as bf16", "*scale = oracle_f32_to_f16(s);", "*scale = oracle_f32_to_bf16(s);"),
    ("division by the stored fp16 scale instead of the fp32 absmax",
     "float r_lo = w[2 * j] / s;\n            float r_hi = w[2 * j + 1] / s;",
     "float r_lo = w[2 * j] / oracle_f16_to_f32(*scale);\n            float r_hi = w[2 * j + 1] / oracle_f16_to_f32(*scale);"),
    ("dequantized value truncated instead of rounded to bf16",
     "return oracle_f32_to_bf16(p);", "uint32_t pb; memcpy(&pb, &p, 4); return (uint16_t)(pb >> 16);"),
    ("dequant product rounded once from double",
     "float p = NF4_TABLE[c] * oracle_f16_to_f32(scale);",
     "float p = (float)((double)NF4_TABLE[c] * (double)oracle_f16_to_f32(scale) * (1.0 + 1e-7));"),
    ("group stride off by one",
     "w_hat[n * K + k] = dequant_value(code_at(codes, K, n, k), scales[n * G + k / NF4_GROUP]);",
     "w_hat[n * K + k] = dequant_value(code_at(codes, K, n, k), scales[n * G + (k > 0 ? k - 1 : 0) / NF4_GROUP]);"),
    ("fp16 ties rounded away from zero",
     "if (rem > half || (rem == half && (r & 1u))) r += 1u;", "if (rem >= half) r += 1u;"),
    ("fp16 subnormal quantum off by one", "int32_t qexp = (E > -14 ? E : -14) - 10;",
     "int32_t qexp = (E > -15 ? E : -15) - 10;"),
    ("bf16 truncation", "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;", ""),
    ("bf16 ties rounded up", "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;",
     "if (lower >= 0x8000u) upper += 1u;"),
    ("table literal typo", "0.5626170039176941f,", "0.5627170039176941f,"),
    ("zero group coded 8 instead of 7", "int lo = 7, hi = 7;", "int lo = 8, hi = 8;"),
    ("absmax ignores the sign", "float a = fabsf(w[k]);", "float a = w[k];"),
    ("linear drops the last term", "double p = xrow[k] * wrow[k];",
     "double p = (k == K - 1) ? 0.0 : xrow[k] * wrow[k];"),
    ("linear subtracts", "acc += p;\n                mag += fabs(p);", "acc -= p;\n                mag += fabs(p);"),
    ("linear magnitude without abs", "acc += p;\n                mag += fabs(p);", "acc += p;\n                mag += p;"),
    ("embed reads the row of the position, not of the id",
     "out[i * K + k] = dequant_value(code_at(codes, K, id, k), scales[id * G + k / NF4_GROUP]);",
     "out[i * K + k] = dequant_value(code_at(codes, K, i % V, k), scales[(i % V) * G + k / NF4_GROUP]);"),
    ("embed writes ones for an id outside the table", "if (id < 0 || id >= V)\n                out[i * K + k] = 0;",
     "if (id < 0 || id >= V)\n                out[i * K + k] = 0x3F80;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation target not found: {old!r}"
    mutated = src.replace(old, new, 1)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.build(str(path), str(tmp_path / "libmutant.so"), force=True)
    o = oracle.Oracle(lib)
    failures = []
    for pin in P.FAST_PINS:
        try:
            pin(o)
        except AssertionError as e:
            failures.append(pin.__name__)
    assert failures, f"no pin caught the planted mistake '{name}'"
