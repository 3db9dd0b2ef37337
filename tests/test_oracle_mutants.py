"""Mutation checks of the oracle's pins (CPU only).

Each case copies oracle/lmoe_oracle.c, plants one plausible mistake in the copy (a wrong
constant, exponent bias or rounding, a dropped term, a swapped operand or index, a flipped
sign or tie-break), builds it with the oracle's own compiler flags, and runs the pin files
that cover that step against the mutant (the oracle package loads the library named by
oracle.LIB_ENV).  The pins must fail: a mistake they let through would be a gap in what pins
the oracle to the pages and the mathematics.  A control case builds the unmodified copy the
same way and must pass the same files.
"""
import os
import shutil
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "lmoe_oracle.c")
HDR = os.path.join(ROOT, "oracle", "lmoe_oracle.h")

FORMATS = ["tests/test_oracle_formats.py"]
QUANT = ["tests/test_oracle_quant.py"]
QUANT2D = ["tests/test_oracle_quant2d.py"]
ROUTER = ["tests/test_oracle_router.py"]
LAYER = ["tests/test_oracle_layer.py"]
SHARED = ["tests/test_oracle_shared.py"]
W4A16 = ["tests/test_oracle_w4a16.py"]

# (name, text in lmoe_oracle.c (unique), its replacement, pin files that must catch it)
MUTANTS = [
    ("e2m1_exponent_bias",
     "ldexp(1.0 + 0.5 * m, e - 1);", "ldexp(1.0 + 0.5 * m, e);", FORMATS),
    ("e2m1_ties_away_from_zero",
     "double q = (a < 2.0) ? 0.5 : (a < 4.0 ? 1.0 : 2.0);\n    double r = nearbyint(a / q) * q;",
     "double q = (a < 2.0) ? 0.5 : (a < 4.0 ? 1.0 : 2.0);\n    double r = floor(a / q + 0.5) * q;", FORMATS),
    ("e4m3_exponent_bias",
     "return sign | (uint8_t)(((E + 7) << 3) | m);", "return sign | (uint8_t)(((E + 8) << 3) | m);", FORMATS),
    ("bf16_nine_significant_bits",
     "int qe = (e - 1) - 7;", "int qe = (e - 1) - 8;", FORMATS),
    ("nvfp4_tensor_scale_without_e2m1_max",
     "const float S = 2688.0f;\n    float s_enc = S / amax;\n    float s_dec = amax / S;\n    quant_job j",
     "const float S = 448.0f;\n    float s_enc = S / amax;\n    float s_dec = amax / S;\n    quant_job j", QUANT),
    ("nvfp4_nibble_order",
     "codes[8 * b + i / 2] = (uint8_t)(q0 | (q1 << 4));", "codes[8 * b + i / 2] = (uint8_t)(q1 | (q0 << 4));",
     QUANT),
    ("nvfp4_block_dot_factor",
     "acc += (double)dot * 0.25 * g_e4m3[sfa[b]] * g_e4m3[sfb[b]];",
     "acc += (double)dot * 0.5 * g_e4m3[sfa[b]] * g_e4m3[sfb[b]];", QUANT),
    ("nvfp4_2d_amax_over_half_the_rows",
     "for (int r = 0; r < 16; ++r)\n                for (int i = 0; i < 16; ++i) {",
     "for (int r = 0; r < 8; ++r)\n                for (int i = 0; i < 16; ++i) {", QUANT2D),
    ("router_ties_to_higher_index",
     "if (best < 0 || lg[e] > lg[best]) best = e;", "if (best < 0 || lg[e] >= lg[best]) best = e;", ROUTER),
    ("router_weights_not_normalised",
     "double v = exp((double)lg[idx[j]] - m) / s;", "double v = exp((double)lg[idx[j]] - m);", ROUTER),
    ("router_logit_unfused_multiply_add",
     "for (int i = c; i < c + 64; ++i) p = fmaf(x[i], w[i], p);",
     "for (int i = c; i < c + 64; ++i) p = p + x[i] * w[i];", ROUTER),
    ("layer_down_projection_transposed",
     "for (int i = 0; i < d; ++i) s += (double)xt[i] * (double)wr[i];\n            z64[j]",
     "for (int i = 0; i < d; ++i) s += (double)xt[i] * (double)L->w_down[(int64_t)i * l + j];\n            z64[j]",
     LAYER),
    ("layer_latent_up_without_relu",
     "L->w1_sf[e] + (int64_t)f * (l / 16), l);\n                    double r = u > 0.0 ? u : 0.0;\n"
     "                    hf[f] = (float)oracle_round_bf16(r * r);\n                    if (hf[f] > hmax)",
     "L->w1_sf[e] + (int64_t)f * (l / 16), l);\n                    double r = u;\n"
     "                    hf[f] = (float)oracle_round_bf16(r * r);\n                    if (hf[f] > hmax)", LAYER),
    ("layer_combine_without_routing_weight",
     "L->w2_sf[e] + (int64_t)j * (F / 16), F);\n                    c64[j] += w64[jj] * o;\n                }\n                if (O->hq_codes)",
     "L->w2_sf[e] + (int64_t)j * (F / 16), F);\n                    c64[j] += o;\n                }\n                if (O->hq_codes)",
     LAYER),
    ("layer_shared_output_subtracted",
     "s += ss64[j];", "s -= ss64[j];", SHARED),
    ("shared_up_without_relu",
     "double u = a1 * oracle_fp8_dot(xq, L->ws1_codes + (int64_t)f * d, d);\n            double r = u > 0.0 ? u : 0.0;",
     "double u = a1 * oracle_fp8_dot(xq, L->ws1_codes + (int64_t)f * d, d);\n            double r = u;", SHARED),
    ("fp8_scale_from_wrong_maximum",
     "fp8_job j = {src, 448.0f / amax, codes};", "fp8_job j = {src, 240.0f / amax, codes};", SHARED),
    ("w4a16_block_scale_dropped",
     "acc += blk * g_e4m3[sfb[b]];", "acc += blk;", W4A16),
    ("w4a16_h_not_rounded_to_bf16",
     "hf[f] = (float)oracle_round_bf16(r * r);\n                }\n                for (int j = 0; j < l; ++j) {\n"
     "                    double o = (double)L->w2_sdec[e] *",
     "hf[f] = (float)(r * r);\n                }\n                for (int j = 0; j < l; ++j) {\n"
     "                    double o = (double)L->w2_sdec[e] *", W4A16),
    ("e4m3_subnormal_spacing",
     "q = ldexp(1.0, -9);", "q = ldexp(1.0, -10);", FORMATS),
    ("bf16_overflow_threshold",
     "const double bf16_max = ldexp(255.0 / 128.0, 127);", "const double bf16_max = ldexp(254.0 / 128.0, 127);",
     FORMATS),
    ("router_slots_in_rank_order",
     "if (taken[e]) idx[n++] = e;", "if (taken[e]) idx[n++] = sel[n];", ROUTER),
    ("router_counts_drop_the_last_slot",
     "for (int64_t i = 0; i < T * k; ++i) counts[idx[i]]++;",
     "for (int64_t i = 0; i + 1 < T * k; ++i) counts[idx[i]]++;", ROUTER),
    ("layer_router_bias_dropped",
     "(L->b_router ? L->b_router[e] : 0.0f);", "0.0f;", LAYER),
    ("layer_z_quantized_with_a_per_token_amax",
     "oracle_quantize_nvfp4(zf, 1, l, J->amax_z, zc, zs, &sd, 1);",
     "oracle_quantize_nvfp4(zf, 1, l, -1.0f, zc, zs, &sd, 1);", LAYER),
    ("layer_h_requantized_with_the_z_scale",
     "oracle_quantize_nvfp4(hf, 1, F, J->amax_h, hc, hs, NULL, 1);",
     "oracle_quantize_nvfp4(hf, 1, F, J->amax_z, hc, hs, NULL, 1);", LAYER),
    ("layer_c_not_rounded_to_bf16",
     "cin[j] = J->quant ? oracle_round_bf16(c64[j]) : c64[j];", "cin[j] = c64[j];", LAYER),
    ("layer_up_projection_transposed",
     "for (int i = 0; i < l; ++i) s += cin[i] * (double)wr[i];",
     "for (int i = 0; i < l; ++i) s += cin[i] * (double)L->w_up[(int64_t)i * d + j];", LAYER),
    ("fp8_dot_units",
     "return ldexp((double)acc, -18);", "return ldexp((double)acc, -17);", SHARED),
    ("e2m1_saturates_to_four",
     "if (!(a < 6.0)) return sign | 7;", "if (!(a < 6.0)) return sign | 6;", FORMATS),
    ("nvfp4_block_amax_without_abs",
     "float a = fabsf(xb[i]);", "float a = xb[i];", QUANT),
    ("nvfp4_2d_scale_on_the_first_row_only",
     "j->sf[(g * 16 + r) * (K / 16) + b] = s;", "if (r == 0) j->sf[(g * 16 + r) * (K / 16) + b] = s;", QUANT2D),
    ("router_groups_of_eight_chunks",
     "for (int g = 0; g < d; g += 16 * 64) {\n        float gs = 0.0f;\n        for (int c = g; c < g + 16 * 64 && c < d; c += 64) {",
     "for (int g = 0; g < d; g += 8 * 64) {\n        float gs = 0.0f;\n        for (int c = g; c < g + 8 * 64 && c < d; c += 64) {",
     ROUTER),
    ("router_flat_sum_of_chunks",
     "            gs = gs + p;\n        }\n        acc = acc + gs;",
     "            acc = acc + p;\n        }\n        (void)gs;", ROUTER),
    ("layer_z_not_rounded_to_bf16",
     "z64[j] = J->quant ? oracle_round_bf16(s) : s;", "z64[j] = s;", LAYER),
    ("layer_y_not_rounded_to_bf16",
     "if (O->y) O->y[t * d + j] = (float)(J->quant ? oracle_round_bf16(s) : s);",
     "if (O->y) O->y[t * d + j] = (float)s;", LAYER),
    ("w4a16_low_nibble_read_as_high",
     "blk += (double)a[16 * b + 2 * i] * (0.5 * g_e2m1x2[c & 15]) +",
     "blk += (double)a[16 * b + 2 * i] * (0.5 * g_e2m1x2[c >> 4]) +", W4A16),
    ("calibration_amax_z_signed",
     "float v = (float)fabs(oracle_round_bf16(s));", "float v = (float)oracle_round_bf16(s);", LAYER),
    ("calibration_amax_h_from_the_unquantized_layer",
     "J.L = &Lc; J.x = x; J.quant = 1; J.out = &none;", "J.L = &Lc; J.x = x; J.quant = 0; J.out = &none;", LAYER),
    ("calibration_shared_amax_x_signed",
     "float a = fabsf(x[i]);", "float a = x[i];", SHARED),
    ("shared_h_quantized_with_the_x_scale",
     "oracle_quantize_fp8(hf, F, amax_hs, hq, &sdh, 1);", "oracle_quantize_fp8(hf, F, amax_xs, hq, &sdh, 1);",
     SHARED),
]


def _build_variant(tmp_path, text):
    d = tmp_path / "src"
    d.mkdir()
    shutil.copy(HDR, d / "lmoe_oracle.h")
    src = d / "lmoe_oracle.c"
    src.write_text(text)
    return oracle.build(force=True, src=str(src), out=str(tmp_path / "liboracle_variant.so"))


def _run_pins(lib_path, files):
    env = dict(os.environ)
    env[oracle.LIB_ENV] = lib_path
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu", *files]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_mutation_sites_are_unique():
    text = open(SRC).read()
    for name, before, _, _ in MUTANTS:
        assert text.count(before) == 1, name


def test_unmodified_copy_passes_the_pins(tmp_path):
    lib = _build_variant(tmp_path, open(SRC).read())
    files = sorted({f for *_, fs in MUTANTS for f in fs})
    r = _run_pins(lib, files)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.parametrize("name,before,after,files", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, before, after, files):
    text = open(SRC).read()
    assert text.count(before) == 1
    lib = _build_variant(tmp_path, text.replace(before, after))
    r = _run_pins(lib, files)
    # exit status 1: the run completed and at least one pin failed (a crash would be another status)
    assert r.returncode == 1, f"mutant {name} passed the pins:\n" + r.stdout[-3000:] + r.stderr[-2000:]
