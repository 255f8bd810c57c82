"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of oracle/q4k_ref.c (on the CPU only),
builds it, and runs the pin suite tests/test_oracle.py against that build; the
suite must fail.  This shows that a dropped term, a wrong sign, index or operand
anywhere in the oracle would not go unnoticed.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "q4k_ref.c")

MUTANTS = {
    "nibble_order_swapped": ("return high ? (b >> 4) : (b & 15);", "return high ? (b & 15) : (b >> 4);"),
    "d_dmin_swapped": ("float d = q4k_ref_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));",
                       "float d = q4k_ref_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));"),
    "high_pair_scale_bits": ("*sc = (scales[j + 4] & 15) | ((scales[j - 4] >> 6) << 4);",
                             "*sc = (scales[j + 4] & 15) | ((scales[j] >> 6) << 4);"),
    "high_pair_min_nibble": ("*m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);",
                             "*m = (scales[j + 4] & 15) | ((scales[j] >> 6) << 4);"),
    "min_sign": ("out[i] = a - b;", "out[i] = a + b;"),
    "sub_block_index": ("int s = i / 32;", "int s = i / 64;"),
    "group_index": ("int g = i / 64;", "int g = i / 32 % 4;"),
    "dropped_last_k": ("for (int64_t k = 0; k < K; ++k) acc +=", "for (int64_t k = 0; k < K - 1; ++k) acc +="),
    "x_row_stride": ("const double *xm = xd + m * K;", "const double *xm = xd + m;"),
    "moe_x_mode": ("(j->x_per_slot ? i : t)", "(j->x_per_slot ? t : i)"),
    "combine_gate_index": ("(double)gates[t * topk + j]", "(double)gates[t * topk]"),
    "route_histogram_offset": ("offsets[ids[i] + 1] += 1;", "offsets[ids[i]] += 1;"),
    "f16_subnormal_scale": ("v = ldexpf((float)f, -24);", "v = ldexpf((float)f, -25);"),
    "bf16_ties_away": ("(lower == 0x8000 && (upper & 1))", "(lower == 0x8000)"),
    "f64_bf16_seven_bits": ("nearbyint(ldexp(m, 8))", "nearbyint(ldexp(m, 7))"),
    "ffn_no_silu": ("g[i] / (1.0 + exp(-g[i])) * u[i]", "g[i] * u[i]"),
    "ffn_down_reads_token_rows": ("rc = q4k_ref_moe_slots(w_down, E, D, H, h, 1, ids, T, topk, out, threads);",
                                  "rc = q4k_ref_moe_slots(w_down, E, D, H, h, 0, ids, T, topk, out, threads);"),
    "x8_ties_away": ("if (a > 0.0f) r = rintf(", "if (a > 0.0f) r = roundf("),
    "x8_scale_128": ("const float sc = a / 127.0f;", "const float sc = a / 128.0f;"),
    "x8_signed_max": ("const float v = fabsf(q4k_ref_bf16_to_f32(xb[i]));", "const float v = q4k_ref_bf16_to_f32(xb[i]);"),
    "x8_scale_block": ("(double)s[m * (K / 32) + k / 32]", "(double)s[m * (K / 32) + ((k / 32) ^ 1)]"),
    "nvfp4_e4m3_bias": ("else v = ldexpf((float)(8 + m), e - 10);", "else v = ldexpf((float)(8 + m), e - 9);"),
    "nvfp4_e2m1_subnormal": ("e == 0 ? 0.5f * (float)m", "e == 0 ? 1.0f * (float)m"),
    "nvfp4_scale_group": ("q4k_ref_e4m3_to_f32(blk[i / 16]) * q4k_ref_e2m1_to_f32(code); /* exact */",
                          "q4k_ref_e4m3_to_f32(blk[i / 32]) * q4k_ref_e2m1_to_f32(code); /* exact */"),
    "nvfp4_nibble_order": ("(i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);\n        const float sv",
                           "(i & 1) ? (uint8_t)(byte & 15) : (uint8_t)(byte >> 4);\n        const float sv"),
    "nvfp4_gemm_no_global": ("wrow[b * QK + i] = j->g * (double)", "wrow[b * QK + i] = (double)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut = tmp_path / "q4k_ref.c"
    mut.write_text(src.replace(old, new))
    (tmp_path / "q4k_ref.h").write_text(open(os.path.join(ROOT, "oracle", "q4k_ref.h")).read())
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-O2", "-ffp-contract=off",
                           "-fPIC", "-shared", str(mut), "-o", str(so), "-lm", "-lpthread"])
    env = dict(os.environ, Q4K_ORACLE_SO=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"),
                        "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the oracle pins:\n{r.stdout[-2000:]}"
