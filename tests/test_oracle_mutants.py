"""The pins catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/fp8_oracle.c (a dropped term,
a wrong sign, bias or index, a changed tie rule), builds it on the CPU, and runs
the oracle pin suite against it in a subprocess: the suite must fail."""
import os
import subprocess
import sys

import pytest

import oracle
from conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "fp8_oracle.c")

MUTANTS = {
    "ties_away_from_even": ("else c = (lo & 1u) ? up : lo;", "else c = up;"),
    "e4m3_bias_off_by_one": ("return ldexp((double)(8 + m), (int)e - 10);",
                             "return ldexp((double)(8 + m), (int)e - 11);"),
    "e5m2_subnormal_scale": ("if (e == 0) return ldexp((double)m, -16);", "if (e == 0) return ldexp((double)m, -15);"),
    "no_saturation": ("if (saturate) return (uint8_t)(sign | maxc);", "if (0) return (uint8_t)(sign | maxc);"),
    "decode_drops_sign": ("return sign ? -v : v;", "return v;"),
    "amax_signed": ("float a = fabsf(bf16_to_float(x[i]));", "float a = bf16_to_float(x[i]);"),
    "amax_f32_signed": ("float a = fabsf(x[i]);", "float a = x[i];"),
    "scale_inverted": ("        s = orc_fmax(fmt) / amax;", "        s = amax / orc_fmax(fmt);"),
    "scale_zero_rule": ("if (!(amax > 0.0f) || isinf(amax)) {", "if (isinf(amax)) {"),
    "history_window_one_slot": ("for (int32_t i = 0; i < len; ++i)\n        if (hist[i] > m)",
                                "for (int32_t i = 0; i < 1; ++i)\n        if (hist[i] > m)"),
    "mx_exponent_strict": ("if ((double)amax <= ldexp(fmax, e)) return e;", "if ((double)amax < ldexp(fmax, e)) return e;"),
    "mx_scale_sign": ("orc_mx_exponent(orc_amax_bf16(blk, 32), fmt);\n            float scale = pow2_neg(e);",
                      "orc_mx_exponent(orc_amax_bf16(blk, 32), fmt);\n            float scale = pow2_neg(-e);"),
    "tile128_first_row_only": ("for (int64_t i = 0; i < 128; ++i) {\n                float a = orc_amax_bf16(",
                               "for (int64_t i = 0; i < 1; ++i) {\n                float a = orc_amax_bf16("),
    # binary32-input quantizers
    "f32_read_through_bf16": ("return orc_encode(x * scale, fmt, 1);",
                              "return orc_encode(bf16_to_float((uint16_t)(float_to_bits(x) >> 16)) * scale, fmt, 1);"),
    "f32_tile128_first_row_only": ("for (int64_t i = 0; i < 128; ++i) {\n                float a = orc_amax_f32(",
                                   "for (int64_t i = 0; i < 1; ++i) {\n                float a = orc_amax_f32("),
    "f32_1x128_block_stride": ("const float* blk = x + r * C + b * 128;", "const float* blk = x + r * C + b * 127;"),
    "f32_mx_scale_sign": ("orc_mx_exponent(orc_amax_f32(blk, 32), fmt);\n            float scale = pow2_neg(e);",
                          "orc_mx_exponent(orc_amax_f32(blk, 32), fmt);\n            float scale = pow2_neg(-e);"),
    # floor-rule MX exponent
    "mx_floor_strict": ("if (ldexp(1.0, e + emax) <= (double)amax) return e;", "if (ldexp(1.0, e + emax) < (double)amax) return e;"),
    "mx_floor_emax": ("int emax = fmt == ORC_E4M3 ? 8 : 15;", "int emax = fmt == ORC_E4M3 ? 9 : 15;"),
    "f32_transpose_index": ("for (int64_t c = 0; c < C; ++c) xt[c * R + r] = x[r * C + c];\n}\n\n/* Plain transpose of a row-major [R, C] bf16",
                            "for (int64_t c = 0; c < C; ++c) xt[c * R + r] = x[c * R + r];\n}\n\n/* Plain transpose of a row-major [R, C] bf16"),
    "dequant_1x128_index": ("case 1: m = (double)sf[r * (C / 128) + c / 128]; break;",
                            "case 1: m = (double)sf[(r / 128) * (C / 128) + c / 128]; break;"),
    "dequant_mx_bias": ("m = e == 255 ? NAN : ldexp(1.0, e - 127);", "m = e == 255 ? NAN : ldexp(1.0, e - 128);"),
    "allreduce_drops_last_rank": ("for (int32_t r = 0; r < k; ++r) acc = acc +", "for (int32_t r = 0; r < k - 1; ++r) acc = acc +"),
    "allreduce_local_amax": ("const float a = orc_amax_bf16(g, (int64_t)k * n);", "const float a = orc_amax_bf16(g, n);"),
    "bf16_ties_away": ("if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;", "if (frac >= 0.5) n += 1.0;"),
    "bf16_subnormal_spacing": ("if (ex < -126) ex = -126;", "if (ex < -127) ex = -127;"),
    "bf16_overflow_early": ("if (res >= ldexp(1.0, 128)) return", "if (res >= ldexp(1.0, 127)) return"),
    "mx_nan_byte_ignored": ("                m = e == 255 ? NAN : ldexp(1.0, e - 127);\n                break;\n            }\n            }\n            out[r * C + c] = v * m;",
                            "                m = ldexp(1.0, e - 127);\n                break;\n            }\n            }\n            out[r * C + c] = v * m;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", *oracle.CFLAGS, str(src), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, FP8_ORACLE_LIB=str(lib))
    out = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_scaling.py"),
                          os.path.join(ROOT, "tests", "test_oracle_formats.py"),
                          os.path.join(ROOT, "tests", "test_oracle_dequant.py"),
                          os.path.join(ROOT, "tests", "test_oracle_allreduce.py"),
                          os.path.join(ROOT, "tests", "test_oracle_f32.py"),
                          os.path.join(ROOT, "tests", "test_oracle_mx_floor.py")],
                         capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
    assert out.returncode != 0, f"the pins did not catch mutant {name}"
