"""Planted mistakes in the oracle must each fail one of its pins (CPU).

Every mutant is one plausible slip: a tie rule, a saturation bound, the sign
of a zero code, the 448 divisor, the scale of an all-zero group, the E4M3
exponent bias or subnormal grid, a mantissa carry, a transposed scale or
code index, a dropped K block, a bfloat16 rounding tie, an amax without the
absolute value; in the Python layer, the dispatch's token order and expert
ids, the expert of a boundary row, the padding of short token groups and the
per-expert scale slice of the grouped Wgrad; for E5M6, the exponent bias,
saturation bound, subnormal grid, mantissa width, sign of zero, divisor,
scale index, amax and the nibble order of the packed layout; for the
power-of-two scales, a non-minimal exponent, the clamp, the sign of the
applied exponent and the rows that carry a weight block's exponent.  The C mutants are compiled from
edited copies of oracle/fp8_oracle.c into temporary libraries, and the
oracle's pin tests are run against each in a fresh process (the oracle loads
the library named by FP8FG_ORACLE_LIB); every such run must fail.  The
Python mutants (oracle/__init__.py, oracle/accumulation.py) are loaded from
edited copies and swapped into the pin modules in place of the oracle.

Nothing here touches the unmodified oracle or any GPU.
"""
import concurrent.futures
import importlib.util
import os
import subprocess
import sys
import tempfile

import pytest

from oracle import build as oracle_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle_quant.py", "tests/test_oracle_gemm.py",
        "tests/test_oracle_dispatch.py", "tests/test_oracle_e4m3.py",
        "tests/test_oracle_e5m6.py", "tests/test_oracle_pow2.py"]

# name -> (exact text of fp8_oracle.c, replacement)
C_MUTANTS = {
    "ties_round_up": ("return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;", "return f + 1.0;"),
    # (a bound anywhere in (448, 464] would be equivalent: round to nearest even
    # already takes every value up to the tie at 464 down to 448)
    "saturation_bound": ("if (a >= 448.0) return", "if (a >= 480.0) return"),
    "zero_code_loses_sign": ("return (uint8_t)(sign | (uint8_t)m);",
                             "return (uint8_t)(m == 0.0 ? 0 : (sign | (uint8_t)m));"),
    "divisor_447": ("return amax / 448.0f;", "return amax / 447.0f;"),
    "zero_group_scale": ("if (amax == 0.0f) return 1.0f;", "if (amax == 0.0f) return 0.5f;"),
    "decode_bias_8": ("v = (1.0 + (double)m / 8.0) * ldexp(1.0, E - 7);",
                      "v = (1.0 + (double)m / 8.0) * ldexp(1.0, E - 8);"),
    "subnormal_grid": ("double m = round_half_even(a * 512.0);",
                       "double m = round_half_even(a * 256.0);"),
    "no_mantissa_carry": ("if (m == 8.0) {            /* mantissa carried into the exponent */",
                          "if (m == 9.0) {            /* mantissa carried into the exponent */"),
    "act_scale_transposed": ("sx[kb * M + m] = s;", "sx[m * KB + kb] = s;"),
    "act_amax_without_abs": ("float v = fabsf(bf16_value(g[j]));", "float v = bf16_value(g[j]);"),
    "tokenwise_scale_transposed": ("sxT[mb * K + k] = s;", "sxT[k * MB + mb] = s;"),
    "weight_codes_transposed": ("if (wq) wq[n * K + k] = q;", "if (wq) wq[k * N + n] = q;"),
    "weight_scale_transposed": ("sw[nb * KB + kb] = s;", "sw[kb * NB + nb] = s;"),
    "dropped_k_block": ("for (int64_t kb = 0; kb < KB; ++kb) {\n                double p = 0.0;",
                        "for (int64_t kb = 0; kb + 1 < KB; ++kb) {\n                double p = 0.0;"),
    "block_b_scale_transposed": ("case FO_BSCALE_BLOCK128: return (double)j->sb[(n / 128) * KB + kb];",
                                 "case FO_BSCALE_BLOCK128: return (double)j->sb[kb * NB + n / 128];"),
    "bf16_ties_away": ("if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;",
                       "if (lo >= 0x8000u) hi += 1u;"),
    # E5M6
    "e5m6_decode_bias_16": ("else v = (1.0 + (double)m / 64.0) * ldexp(1.0, E - 15);",
                            "else v = (1.0 + (double)m / 64.0) * ldexp(1.0, E - 16);"),
    "e5m6_saturation_bound": ("if (a >= 65024.0) return (uint16_t)(sign | 0x7BF);",
                              "if (a >= 65536.0) return (uint16_t)(sign | 0x7BF);"),
    "e5m6_subnormal_grid": ("double m = round_half_even(a * 1048576.0);",
                            "double m = round_half_even(a * 2097152.0);"),
    "e5m6_five_mantissa_bits": ("double m = round_half_even((2.0 * fr - 1.0) * 64.0);",
                                "double m = round_half_even((2.0 * fr - 1.0) * 32.0);"),
    "e5m6_zero_code_loses_sign": ("return (uint16_t)(sign | (uint16_t)m);",
                                  "return (uint16_t)(m == 0.0 ? 0 : (sign | (uint16_t)m));"),
    "e5m6_divisor_65536": ("return amax / 65024.0f;", "return amax / 65536.0f;"),
    "e5m6_zero_group_scale": ("if (amax == 0.0f) { return 1.0f; }",
                              "if (amax == 0.0f) { return 0.5f; }"),
    # power-of-two scales
    "pow2_not_minimal": ("while (e < 127 && (double)amax > 448.0 * ldexp(1.0, e)) ++e;",
                         "while (e < 127 && (double)amax >= 448.0 * ldexp(1.0, e)) ++e;"),
    "pow2_clamp_126": ("    int e = -127;\n    while", "    int e = -126;\n    while"),
    "pow2_scale_not_applied": ("xq[m * ldq + kb * 128 + j] = fo_e4m3_encode((float)ldexp((double)bf16_value(src[j]), -e));",
                               "xq[m * ldq + kb * 128 + j] = fo_e4m3_encode((float)ldexp((double)bf16_value(src[j]), e));"),
    "pow2_weight_rows_of_block_0": ("for (int j = 0; j < 128; ++j) se8[kb * N + nb * 128 + j] = (uint8_t)(e + 127);",
                                    "for (int j = 0; j < 128; ++j) se8[kb * N + j] = (uint8_t)(e + 127);"),
    "e5m6_scale_transposed": ("sx[m + kb * M] = s;", "sx[m * KB + kb] = s;"),
    "e5m6_amax_without_abs": ("float mag = fabsf(bf16_value(grp[j]));",
                              "float mag = bf16_value(grp[j]);"),
}


def _compile(src_text, out_path):
    with tempfile.NamedTemporaryFile("w", suffix=".c", delete=False) as f:
        f.write(src_text)
        c_path = f.name
    try:
        subprocess.run(["gcc", *oracle_build.CFLAGS, c_path, "-o", out_path, "-lm"], check=True,
                       capture_output=True)
    finally:
        os.unlink(c_path)


def _run_pins(lib_path):
    env = dict(os.environ, FP8FG_ORACLE_LIB=lib_path, OMP_NUM_THREADS="4")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu",
                        "-p", "no:cacheprovider", *PINS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-400:]


def test_every_c_mutant_fails_a_pin(tmp_path):
    src = open(oracle_build.SRC).read()
    libs = {}
    for name, (old, new) in C_MUTANTS.items():
        assert src.count(old) == 1, "mutant %s: pattern not unique in fp8_oracle.c" % name
        lib = str(tmp_path / ("lib_%s.so" % name))
        _compile(src.replace(old, new), lib)
        libs[name] = lib
    # the unmodified source, built the same way, passes the same pins
    clean = str(tmp_path / "lib_clean.so")
    _compile(src, clean)
    rc, out = _run_pins(clean)
    assert rc == 0, "unmodified oracle fails its pins:\n" + out
    with concurrent.futures.ThreadPoolExecutor(max_workers=4) as ex:
        results = dict(zip(libs, ex.map(_run_pins, libs.values())))
    survivors = [name for name, (rc, _) in results.items() if rc == 0]
    assert not survivors, "mutants that pass every pin: %s" % survivors
    # a failing run must be a failed assertion, not a crash or a collection error
    for name, (rc, out) in results.items():
        assert rc == 1, "mutant %s: pytest exit %d\n%s" % (name, rc, out)


# ------------------------------------------------ accumulation model --------
ACC_MUTANTS = {
    "nearest_instead_of_truncation": ("np.trunc(np.ldexp(m, bits))", "np.rint(np.ldexp(m, bits))"),
    "no_restart_after_promotion": ("            tc = np.zeros((M, N), np.float64)\n",
                                   "            pass\n"),
    "b_scale_transposed": ("sb[nb_of_col, kb]",
                           "sb[kb % sb.shape[0], np.minimum(nb_of_col, sb.shape[1] - 1)]"),
    "cut_before_the_add": ("tc = truncate_significand(tc + step, bits)",
                           "tc = tc + truncate_significand(step, bits)"),
    "one_bit_off": ("np.ldexp(m, bits)), e - bits)", "np.ldexp(m, bits - 1)), e - bits + 1)"),
}


def _acc_module(text, name):
    spec = importlib.util.spec_from_loader("oracle.acc_mutant_" + name, loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    exec(compile(text, "accumulation_" + name, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(ACC_MUTANTS))
def test_every_accumulation_mutant_fails_a_pin(name, monkeypatch):
    import test_oracle_accumulation as pins
    path = os.path.join(ROOT, "oracle", "accumulation.py")
    src = open(path).read()
    old, new = ACC_MUTANTS[name]
    assert src.count(old) == 1, "mutant %s: pattern not unique" % name
    monkeypatch.setattr(pins, "acc", _acc_module(src.replace(old, new), name))
    checks = [pins.test_truncate_against_integer_shifts, pins.test_full_width_is_exact,
              pins.test_hand_worked_narrow_accumulator,
              lambda: pins.test_truncation_error_bounds(14),
              pins.test_promotion_keeps_the_error_flat_in_k]
    failed = 0
    for check in checks:
        try:
            check()
        except AssertionError:
            failed += 1
    assert failed > 0, "accumulation mutant %s passes every pin" % name


# ------------------------------------------------ Python layer of the oracle --
PY_MUTANTS = {  # name -> (exact text of oracle/__init__.py, replacement, pin module, pins)
    "dispatch_tokens_descending": (
        "token_lists = [np.nonzero(member[:, e])[0] for e in range(n_local)]",
        "token_lists = [np.nonzero(member[:, e])[0][::-1] for e in range(n_local)]",
        "test_oracle_dispatch", None),
    "dispatch_expert_ids_off_by_one": (
        "experts = expert_begin + np.arange(n_local, dtype=np.int64)",
        "experts = expert_begin + 1 + np.arange(n_local, dtype=np.int64)",
        "test_oracle_dispatch", None),
    "grouped_boundary_row_to_previous_expert": (
        'expert_of = np.searchsorted(offsets, rows, side="right") - 1',
        'expert_of = np.maximum(np.searchsorted(offsets, rows, side="left") - 1, 0)',
        "test_oracle_gemm", ["test_grouped_equals_dense_per_expert",
                             "test_grouped_dgrad_equals_dequantised_product"]),
    "short_group_padded_with_ones": (
        "seg = np.zeros((padded[e], K), np.uint16)  # bfloat16 +0",
        "seg = np.full((padded[e], K), 0x3F80, np.uint16)",
        "test_oracle_gemm", ["test_grouped_128x1_single_expert_is_the_dense_quantiser",
                             "test_grouped_128x1_short_groups",
                             "test_grouped_wgrad_equals_dequantised_product"]),
    "e5m6_pack_nibbles_swapped": (
        "out[..., 1] = ((c0 >> 8) & 0xF) | ((c1 & 0xF) << 4)",
        "out[..., 1] = (c1 & 0xF) | (((c0 >> 8) & 0xF) << 4)",
        "test_oracle_e5m6", ["test_packing_bit_layout"]),
    "wgrad_b_scales_of_expert_0": (
        "sb[lo // 128:hi // 128], BSCALE_ROW1x128",
        "sb[:hi // 128 - lo // 128], BSCALE_ROW1x128",
        "test_oracle_gemm", ["test_grouped_wgrad_equals_dequantised_product"]),
}


def _oracle_module(text, name):
    spec = importlib.util.spec_from_loader("oracle.mutant_" + name, loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    mod.__path__ = [os.path.join(ROOT, "oracle")]
    exec(compile(text, "oracle_" + name, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_every_python_oracle_mutant_fails_a_pin(name, monkeypatch):
    old, new, module, names = PY_MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert src.count(old) == 1, "mutant %s: pattern not unique" % name
    pins = importlib.import_module(module)
    monkeypatch.setattr(pins, "oracle", _oracle_module(src.replace(old, new), name))
    if names is None:
        names = [n for n in dir(pins) if n.startswith("test_")]
    failed = 0
    for n in names:
        try:
            getattr(pins, n)()
        except AssertionError:
            failed += 1
    assert failed > 0, "oracle mutant %s passes every pin" % name


def test_harness_passes_with_the_unmodified_sources(monkeypatch):
    """Controls: unmodified copies loaded the same way pass every pin used above."""
    import test_oracle_accumulation as acc_pins
    src = open(os.path.join(ROOT, "oracle", "accumulation.py")).read()
    monkeypatch.setattr(acc_pins, "acc", _acc_module(src, "clean"))
    for check in [acc_pins.test_truncate_against_integer_shifts, acc_pins.test_full_width_is_exact,
                  acc_pins.test_hand_worked_narrow_accumulator,
                  lambda: acc_pins.test_truncation_error_bounds(14),
                  acc_pins.test_promotion_keeps_the_error_flat_in_k]:
        check()
    src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    for module in ("test_oracle_dispatch", "test_oracle_gemm", "test_oracle_e5m6"):
        pins = importlib.import_module(module)
        monkeypatch.setattr(pins, "oracle", _oracle_module(src, "clean"))
        names = {n for _, _, m, ns in PY_MUTANTS.values() if m == module
                 for n in (ns or [x for x in dir(pins) if x.startswith("test_")])}
        for n in sorted(names):
            getattr(pins, n)()
