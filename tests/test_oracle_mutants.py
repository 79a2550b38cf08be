"""The oracle's pins have teeth: plant one plausible mistake at a time in a
copy of ``oracle/oracle.c`` (on the CPU), build the copy, and check that the
pin suite fails against it.  The real oracle is never modified."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

PINS = "test_oracle_pins.py"
ATTN_PINS = "test_oracle_attention_pins.py"
LAYOUT_PINS = "test_oracle_layout_pins.py"
FP8_PINS = "test_oracle_fp8_pins.py"

# (name, text to replace, replacement, count[, pins file]) -- each must occur in oracle.c
MUTANTS = [
    ("drop_last_k", "for (int64_t k = 0; k < K; ++k) {\n                    double b",
     "for (int64_t k = 0; k < K - 1; ++k) {\n                    double b", 1),
    ("transposed_B_index", "lut[B[k + n * K]]", "lut[B[n + k * N]]", 1),
    ("f16_sign_dropped", "v = ldexp((double)(1024 + f), e - 25);  /* (1.f) * 2^(e-15) */\n    }\n    return sign ? -v : v;",
     "v = ldexp((double)(1024 + f), e - 25);  /* (1.f) * 2^(e-15) */\n    }\n    return v;", 1),
    ("truncate_not_round", "double n = rint(ldexp(a, frac_bits - E));",
     "double n = floor(ldexp(a, frac_bits - E));", 1),
    ("bf16_wrong_bias", "e - 134", "e - 133", 1),
    ("bf16_double_rounding", "return orc_round_to_format(x, 7, 127, 255);",
     "return orc_round_to_format((double)(float)x, 7, 127, 255);", 1),
    ("linear_reversed_k", "acc += xr[k] * lut[wrow[k]];", "acc += xr[k] * lut[wrow[K - 1 - k]];", 2),
    ("f32_accumulator", "double* acc = (double*)malloc", "float* acc = (float*)malloc", 2),
    ("attn_drop_last_token", "for (int64_t t = 0; t < L; ++t) {\n                    const int64_t blk",
     "for (int64_t t = 0; t < L - 1; ++t) {\n                    const int64_t blk", 1, ATTN_PINS),
    ("attn_wrong_group", "const int64_t g = h / group;", "const int64_t g = h % num_kv_heads;", 1, ATTN_PINS),
    ("attn_no_max_subtraction", "const double p = exp(sc[t] - mx);", "const double p = exp(sc[t]);", 1, ATTN_PINS),
    ("attn_wrong_block_offset", "((blk * block_size + t % block_size) * num_kv_heads + g) * hd",
     "((blk * block_size + t / block_size) * num_kv_heads + g) * hd", 1, ATTN_PINS),
    ("attn_ignores_scale", "sc[t] = scale * d;", "sc[t] = d;", 1, ATTN_PINS),
    ("general_transb_ignored", "int64_t bi = transb ? orc_at(row_major, n, k, ldb) : orc_at(row_major, k, n, ldb);",
     "int64_t bi = orc_at(row_major, k, n, ldb);", 1, LAYOUT_PINS),
    ("general_row_major_swapped", "return row_major ? c + r * ld : r + c * ld;",
     "return row_major ? r + c * ld : c + r * ld;", 1, LAYOUT_PINS),
    ("general_lda_ignored", "orc_at(row_major, k, m, lda) : orc_at(row_major, m, k, lda)",
     "orc_at(row_major, k, m, K) : orc_at(row_major, m, k, M)", 1, LAYOUT_PINS),
    ("general_bias_first_only", "v += lut[bias[m]];", "v += lut[bias[0]];", 1, LAYOUT_PINS),
    ("general_bias_after_rounding", "if (out) out[i + j * nr] = orc_f16_encode_rn(v);",
     "if (out) out[i + j * nr] = orc_f16_encode_rn(lut[orc_f16_encode_rn(acc[i])] + (v - acc[i]));", 1,
     LAYOUT_PINS),
    ("fp8_e4m3_wrong_bias", "else v = ldexp((double)(8 + f), e - 10);", "else v = ldexp((double)(8 + f), e - 11);", 1,
     FP8_PINS),
    ("fp8_e4m3_ieee_nan_rule", "else if (e == 15 && f == 7) v = NAN;", "else if (e == 15) v = NAN;", 1, FP8_PINS),
    ("fp8_e5m2_subnormal_scale", "if (e == 0) v = ldexp((double)f, -16);", "if (e == 0) v = ldexp((double)f, -15);", 1,
     FP8_PINS),
    ("fp8_alpha_ignored", "double v = alpha * acc;", "double v = acc;", 1, FP8_PINS),
    ("fp8_reversed_b", "acc += lut[a_row[k]] * lut[b_col[k]];", "acc += lut[a_row[k]] * lut[b_col[K - 1 - k]];", 1,
     FP8_PINS),
    ("f32_wrong_sign_bit", "return orc_round_bits(x, 23, 127, 255, 31);", "return orc_round_bits(x, 23, 127, 255, 15);",
     1, FP8_PINS),
    ("fp8_bf16_double_rounding", "out16[i + j * nr] = orc_bf16_encode_rn(v);",
     "out16[i + j * nr] = orc_bf16_encode_rn((double)(float)v);", 1, FP8_PINS),
]


@pytest.mark.slow
@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, mutant):
    name, old, new, count = mutant[:4]
    pins = mutant[4] if len(mutant) > 4 else PINS
    src = open(SRC).read()
    assert src.count(old) == count, f"mutant {name}: pattern not found as expected"
    mutated = src.replace(old, new)
    if name == "f32_accumulator":
        mutated = mutated.replace("(size_t)(M > 0 ? M : 1) * sizeof(double)", "(size_t)(M > 0 ? M : 1) * sizeof(float)")
    csrc = tmp_path / "oracle_mutant.c"
    csrc.write_text(mutated)
    lib = tmp_path / "liboracle_mutant.so"
    r = subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", str(csrc), "-o", str(lib), "-lm"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", pins)],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
