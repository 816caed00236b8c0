"""The oracle's pins have teeth: plant one plausible mistake at a time in a
temporary copy of the oracle source (on the CPU), build it, and check that at
least one pin from the oracle test files fails on it.

Mistakes planted: a wrong sign, a dropped term, a transposed or wrong
operand, a wrong row index for a broadcast operand, eps outside the root or
dropped, a wrong divisor in the mean, a fused multiply-add, wrong rounding of
the storage dtype, the fused op reading the unrounded residual; in the row
statistic a double-precision sum, truncation, ties away from zero, squares
cut to fp32 precision and a doubly rounded inverse root; and in the
GELU a wrong coefficient, power, sign or scale, and double rounding; in the
FP8 output the scale applied the wrong way, no saturation, ties away from
zero and a wrong subnormal spacing.
"""
import os
import shutil
import subprocess

import pytest

import oracle
import test_oracle_codecs as pc
import test_oracle_fp8 as p8
import test_oracle_fused as pf
import test_oracle_gelu as pg
import test_oracle_modulate as pm
import test_oracle_residual_gate as pr
import test_oracle_statistic as ps

SRC = os.path.join(os.path.dirname(oracle.__file__), "dit_oracle.c")

MUTANTS = {
    "rga_minus": ("float s = h + p;", "float s = h - p;"),
    "rga_wrong_operand": ("float p = u * g;", "float p = h * g;"),
    "rga_fma": ("float p = u * g;\n    float s = h + p;",
                "float p = u * g;\n    float s = fmaf(u, g, h); (void)p;"),
    "rga_bcast_row": ("int64_t grow = (gate_layout == ORC_FULL) ? r : r / L;",
                      "int64_t grow = (gate_layout == ORC_FULL) ? r : r % L;"),
    "mod_shift_sign": ("float y = t + sh;", "float y = t - sh;"),
    "mod_drop_one": ("float one = 1.0f + sc;", "float one = sc;"),
    "mod_swap_scale_shift": ("float sc = orc_load(scale, mrow * D + d, dtype);\n"
                             "    float sh = orc_load(shift, mrow * D + d, dtype);",
                             "float sc = orc_load(shift, mrow * D + d, dtype);\n"
                             "    float sh = orc_load(scale, mrow * D + d, dtype);"),
    "mod_drop_eps": ("float v = ms + eps;", "float v = ms; (void)eps;"),
    "mod_eps_outside": ("  float v = ms + eps;\n  return inverse_root(v);",
                        "  return (float)(1.0 / (sqrt((double)ms) + (double)eps));"),
    "mod_mean_divisor": ("return rn32_mean(digit, (uint32_t)D);",
                         "return rn32_mean(digit, (uint32_t)D + 1);"),
    # the statistic: a double-precision sum (the earlier reading), no
    # rounding, ties away from zero, squares cut to fp32 precision, and the
    # inverse root rounded twice (fp32 root, then fp32 quotient)
    "stat_double_sum": ("  exact_sum_of_squares(x_row, D, dtype, digit);\n"
                        "  return rn32_mean(digit, (uint32_t)D);",
                        "  double s = 0.0; (void)digit;\n"
                        "  for (int64_t d = 0; d < D; ++d) { double v = orc_load(x_row, d, dtype); s += v * v; }\n"
                        "  return (float)(s / (double)D);"),
    "stat_truncate": ("if (guard && (sticky || (mant & 1u))) mant += 1;",
                      "(void)guard; (void)sticky;"),
    "stat_ties_away": ("if (guard && (sticky || (mant & 1u))) mant += 1;",
                       "if (guard) mant += 1; (void)sticky;"),
    "stat_fp32_squares": ("const uint64_t sq = M * M;",
                          "const uint64_t sq = (M * M) >> 24 << 24;"),
    "stat_root_in_fp32": ("static float inverse_root(float v) { return (float)(1.0 / sqrt((double)v)); }",
                          "static float inverse_root(float v) { return 1.0f / sqrtf(v); }"),
    "mod_bcast_row": ("int64_t mrow = (mod_layout == ORC_FULL) ? r : r / L;",
                      "int64_t mrow = (mod_layout == ORC_FULL) ? r : 0;"),
    "bf16_round_half_up": ("x += 0x7FFFu + lsb;", "x += 0x8000u; (void)lsb;"),
    "fp16_truncate": ("float m = nearbyintf(a / ldexpf(1.0f, E - 10));",
                      "float m = truncf(a / ldexpf(1.0f, E - 10));"),
    "fp8_scale_inverted": ("orc_f32_to_e4m3(y * qinv)", "orc_f32_to_e4m3(y / qinv)"),
    "fp8_no_saturation": ("if (a >= 448.0) return sign | 0x7E;",
                          "if (a >= 464.0) return sign | 0x7F;"),
    "fp8_ties_away": ("double k = nearbyint(a / ldexp(1.0, E - 3));",
                      "double k = round(a / ldexp(1.0, E - 3));"),
    "fp8_subnormal_spacing": ("const double k = nearbyint(a / ldexp(1.0, -9));",
                              "const double k = nearbyint(a / ldexp(1.0, -10));"),
    "gelu_cubic_coeff": ("0.044715 * v * v * v", "0.04715 * v * v * v"),
    "gelu_square": ("0.044715 * v * v * v", "0.044715 * v * v"),
    "gelu_sign": ("v / (1.0 + exp(-2.0 * z))", "v / (1.0 + exp(2.0 * z))"),
    "gelu_half_z": ("v / (1.0 + exp(-2.0 * z))", "v / (1.0 + exp(-z))"),
    "double_rounding": ("    b |= 1u; /* sticky: odd */", "    (void)b;"),
    "fused_unrounded": (
        "      rmsnorm_modulate_row(j->out2, j->t_out, j->out, j->scale, j->shift, r,\n"
        "                           j->L, j->D, j->eps, j->dtype, j->layout2, j->fp8, j->qinv);",
        # modulate the fp32 sums instead of the stored (rounded) residual
        "      { float* xr = malloc(sizeof(float) * (size_t)j->D); double sum = 0;\n"
        "        int64_t gr = j->layout1 == ORC_FULL ? r : r / j->L;\n"
        "        int64_t mr = j->layout2 == ORC_FULL ? r : r / j->L;\n"
        "        for (int64_t d = 0; d < j->D; ++d) {\n"
        "          int64_t i = r * j->D + d;\n"
        "          xr[d] = orc_load(j->hidden, i, j->dtype) +\n"
        "                  orc_load(j->update, i, j->dtype) * orc_load(j->gate, gr * j->D + d, j->dtype);\n"
        "          sum += (double)xr[d] * xr[d]; }\n"
        "        float rv = (float)(1.0 / sqrt((double)((float)(sum / j->D) + j->eps)));\n"
        "        for (int64_t d = 0; d < j->D; ++d) {\n"
        "          float t = (xr[d] * rv) * (1.0f + orc_load(j->scale, mr * j->D + d, j->dtype));\n"
        "          orc_store(j->out2, r * j->D + d,\n"
        "                    t + orc_load(j->shift, mr * j->D + d, j->dtype), j->dtype); }\n"
        "        free(xr); }"),
}

# Pins run against each mutant (a fast subset of the oracle test files).
PINS = [
    lambda o: pc.test_rounding_ties_golden(o),
    lambda o: pc.test_bf16_encode_matches_torch(o),
    lambda o: pc.test_fp16_encode_matches_numpy(o),
    lambda o: pr.test_gate_one_is_library_add(o, "bf16", "full"),
    lambda o: pr.test_bcast_equals_expanded_full_gate(o, "bf16"),
    lambda o: pr.test_bcast_batch_permutation(o),
    lambda o: pr.test_worked_examples_golden(o),
    lambda o: pr.test_signed_zero_of_an_underflowing_product(o),
    lambda o: pr.test_exact_rational_bruteforce(o, "bf16", "bcast", (2, 3, 7)),
    lambda o: pr.test_exact_rational_bruteforce(o, "fp32", "full", (2, 3, 7)),
    lambda o: pm.test_zero_modulation_gives_unit_mean_square(o, "bcast"),
    lambda o: pm.test_scale_minus_one_gives_shift(o, "bf16", "bcast"),
    lambda o: pm.test_constant_row_closed_form(o, 1e-3),
    lambda o: pm.test_against_torch_rms_norm_float64(o, "bf16", "bcast"),
    lambda o: pm.test_worked_examples_golden(o),
    lambda o: pm.test_bcast_equals_expanded_and_batches(o, "bf16"),
    lambda o: pf.test_exact_bruteforce(o, "bf16", (2, 2, 16)),
    lambda o: pg.test_round_to_odd_avoids_double_rounding(o),
    lambda o: pg.test_against_torch_float64(o, "bf16"),
    lambda o: pg.test_against_50_digit_evaluation(o, "fp32"),
    lambda o: p8.test_ties_golden(o),
    lambda o: p8.test_encode_against_torch(o),
    lambda o: p8.test_modulate_fp8_is_quantised_fp32_modulation(o, "bf16", 0.005),
    lambda o: [ps.test_mean_square_golden(o, c) for c in ps.parse_golden()],
    lambda o: ps.test_mean_square_matches_exact_rationals(o, "bf16", 7),
    lambda o: ps.test_mean_square_matches_exact_rationals(o, "fp32", 3),
    lambda o: ps.test_inverse_root_across_the_range(o),
]


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    d = tmp_path_factory.mktemp("mutants")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(orc, mutant_dir, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not found for {name}"
    path = mutant_dir / f"{name}.c"
    path.write_text(src.replace(old, new))
    hdr = os.path.join(os.path.dirname(SRC), "dit_oracle.h")
    lib = mutant_dir / f"lib{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-I", os.path.dirname(hdr), "-o", str(lib), str(path), "-lm",
                    "-lpthread"], check=True)
    mut = oracle.variant(str(lib))
    failures = 0
    for pin in PINS:
        try:
            pin(mut)
        except AssertionError:
            failures += 1
    assert failures >= 1, f"no pin caught mutant {name}"


def test_unmutated_copy_passes_every_pin(orc, mutant_dir):
    """Control: the same build route with no mutation fails no pin."""
    lib = mutant_dir / "libcontrol.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(lib), SRC, "-lm", "-lpthread"], check=True)
    ctl = oracle.variant(str(lib))
    for pin in PINS:
        pin(ctl)
