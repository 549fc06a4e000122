"""The oracle's pins catch planted mistakes.

Each case copies the oracle package to a temporary folder, plants ONE
plausible slip in the copy (a wrong constant, a wrong rounding mode, a dropped
term, a wrong sign, a wrong index, a transposed operand), compiles it with the
oracle's own gcc flags and runs the pin files against the copy in a child
process.  The case passes when at least one pin FAILS on the copy; a mutant
that passes every pin would mean the pins cannot tell that mistake from the
definition.  Nothing here touches the committed oracle or any GPU.

The slips, by the passage each one breaks:

* the quantizer ("Realizing Native INT8 Compute for Diffusion Transformers on
  Consumer GPUs", abstract: symmetric per-token / per-channel INT8 with the
  scale absmax / 127 and round-to-nearest codes): 128 for 127, a reciprocal
  multiply, ties away from zero, truncation, max for absmax, a nonzero scale
  for the zero row;
* the int8 x int8 -> int32 GEMM (same abstract): a 16-bit accumulator, a
  dropped last term, a reversed index, the activation squared, transposed
  operands;
* the epilogue (same abstract: per-token x per-channel dequantization plus
  bias, bf16 out): a dropped per-token scale, the channel scale used twice, a
  dropped or negated bias, truncating or ties-away bf16 rounding;
* the E4M3 arm (OCP 8-bit floating point specification, E4M3 encoding:
  bias 7, subnormal spacing 2^-9, largest finite 448, no infinity): each of
  those constants, the rounding mode, the NaN code, the sign of the codes in
  the GEMM, the scale's 448;
* the fused producers (LayerNorm without affine: biased variance, eps inside
  the square root; GELU in its erf form): the unbiased variance, eps outside
  the root, a dropped mean, the tanh approximation, an unscaled erf argument,
  a sign slip in the negative branch, the cancelling 1 + erf form below -8;
  and the single fp64 -> bf16 rounding (ties away, one bit short).
"""
import os
import re
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")
PIN_FILES = ["tests/test_oracle.py", "tests/test_oracle_fp8.py",
             "tests/test_oracle_fused.py"]

C, PY = "i8_oracle.c", "__init__.py"

# (id, file, anchor, old, new): replace the first `old` after `anchor`.
MUTANTS = [
    # quantizer
    ("quant_scale_128", C, "static void quant_one_row(", "amax / 127.0f", "amax / 128.0f"),
    ("quant_reciprocal_multiply", C, "static void quant_one_row(",
     "orc_bf16_to_f32(x[k]) / s;", "orc_bf16_to_f32(x[k]) * (1.0f / s);"),
    ("quant_ties_away", C, "static void quant_one_row(", "rintf(t)", "roundf(t)"),
    ("quant_truncates", C, "static void quant_one_row(", "rintf(t)", "truncf(t)"),
    ("quant_max_not_absmax", C, "static void quant_one_row(",
     "fabsf(orc_bf16_to_f32(x[k]))", "orc_bf16_to_f32(x[k])"),
    ("quant_zero_row_scale_one", C, "static void quant_one_row(",
     "*scale = 0.0f;", "*scale = 1.0f;"),
    # int32 GEMM
    ("gemm_int16_accumulator", C, "int orc_gemm_s32(", "int32_t acc = 0;", "int16_t acc = 0;"),
    ("gemm_drops_last_k", C, "int orc_gemm_s32(",
     "for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k + 1 < K; ++k)"),
    ("gemm_reversed_weight_index", C, "int orc_gemm_s32(",
     "(int32_t)wrow[k]", "(int32_t)wrow[K - 1 - k]"),
    ("gemm_squares_activation", C, "int orc_gemm_s32(",
     "(int32_t)wrow[k]", "(int32_t)arow[k]"),
    ("linear_transposed_operands", PY, "def linear(x_bits",
     "acc = gemm_s32(aq, wq)", "acc = gemm_s32(wq, aq)"),
    # epilogue and bf16 rounding
    ("epi_drops_token_scale", C, "int orc_dequant_bias(", "t = t * s_a[m];", "t = t * 1.0f;"),
    ("epi_channel_scale_twice", C, "int orc_dequant_bias(", "t = t * s_a[m];", "t = t * s_w[n];"),
    ("epi_drops_bias", C, "int orc_dequant_bias(",
     "(bias ? orc_bf16_to_f32(bias[n]) : 0.0f)", "0.0f"),
    ("epi_negates_bias", C, "int orc_dequant_bias(", "t = t + (bias", "t = t - (bias"),
    ("bf16_truncates", C, "uint16_t orc_f32_to_bf16(", "u + 0x7fffu + lsb", "u + 0u * lsb"),
    ("bf16_ties_away", C, "uint16_t orc_f32_to_bf16(", "u + 0x7fffu + lsb", "u + 0x8000u + 0u * lsb"),
    # E4M3 arm
    ("e4m3_scale_240", C, "static void quant_one_row_e4m3(", "amax / 448.0f", "amax / 240.0f"),
    ("e4m3_exponent_bias_8", C, "double orc_e4m3_to_f64(", "e - 10)", "e - 11)"),
    ("e4m3_subnormal_spacing", C, "double orc_e4m3_to_f64(",
     "ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    ("e4m3_encode_ties_away", C, "uint8_t orc_f32_to_e4m3(",
     "nearbyint(a / quantum)", "round(a / quantum)"),
    ("e4m3_saturates_past_448", C, "uint8_t orc_f32_to_e4m3(",
     "if (r > 448.0) r = 448.0;", "if (r > 480.0) r = 480.0;"),
    ("e4m3_nan_code", C, "uint8_t orc_f32_to_e4m3(", "return 0x7F;", "return 0x7E;"),
    ("e4m3_gemm_squares_activation", C, "int orc_gemm_e4m3_f64(",
     "val[wrow[k]]", "val[arow[k]]"),
    ("e4m3_gemm_drops_sign", C, "int orc_gemm_e4m3_f64(",
     "val[b] = absval ? fabs(v) : v;", "val[b] = fabs(v) + 0 * absval;"),
    ("linear_e4m3_transposed_operands", PY, "def linear_e4m3(",
     "acc = gemm_e4m3_f64(aq, wq)", "acc = gemm_e4m3_f64(wq, aq)"),
    # fused producers and the fp64 -> bf16 rounding
    ("f64_bf16_ties_away", C, "uint16_t orc_f64_to_bf16(", "nearbyint(a / q)", "round(a / q)"),
    ("f64_bf16_one_bit_short", C, "uint16_t orc_f64_to_bf16(",
     "ldexp(1.0, lg - 7)", "ldexp(1.0, lg - 6)"),
    ("ln_unbiased_variance", C, "int orc_layernorm_rows(",
     "var /= (double)K;", "var /= (double)(K - 1);"),
    ("ln_eps_outside_sqrt", C, "int orc_layernorm_rows(", "sqrt(var + eps)", "sqrt(var) + eps"),
    ("ln_drops_mean", C, "int orc_layernorm_rows(",
     "((double)orc_bf16_to_f32(xr[k]) - mu) / rs", "((double)orc_bf16_to_f32(xr[k])) / rs"),
    ("gelu_tanh_approximation", C, "int orc_gelu_rows(",
     "v >= 0.0 ? 0.5 * (1.0 + erf(v / sqrt(2.0))) : 0.5 * erfc(-v / sqrt(2.0))",
     "0.5 * (1.0 + tanh(0.7978845608028654 * (v + 0.044715 * v * v * v)))"),
    ("gelu_erf_argument_unscaled", C, "int orc_gelu_rows(", "erf(v / sqrt(2.0))", "erf(v / 2.0)"),
    ("gelu_negative_branch_sign", C, "int orc_gelu_rows(",
     "erfc(-v / sqrt(2.0))", "erfc(v / sqrt(2.0))"),
    ("gelu_cancelling_form", C, "int orc_gelu_rows(",
     "v >= 0.0 ? 0.5 * (1.0 + erf(v / sqrt(2.0))) : 0.5 * erfc(-v / sqrt(2.0))",
     "0.5 * (1.0 + erf(v / sqrt(2.0)))"),
    ("producer_quantizes_its_input", PY, "def producer_quant_rows(",
     "quant_rows(y) if", "quant_rows(x_bits) if"),
]


# The same pipeline with nothing planted: every pin must pass on the copy, so
# that a killed mutant is the planted slip and not the copying or the child run.
CONTROL = ("control_unmodified", C, "static void quant_one_row(", "", "")


def _plant(src: str, anchor: str, old: str, new: str) -> str:
    a = src.index(anchor)
    i = src.index(old, a)
    return src[:i] + new + src[i + len(old):]


def _run_mutant(mutant, workdir):
    """Plant, compile and run the pins; returns (outcome, the first failing
    pin when killed, else the end of the log)."""
    mid, fname, anchor, old, new = mutant
    pkg = os.path.join(workdir, mid, "oracle")
    planted = old != new
    os.makedirs(pkg)
    for f in ("__init__.py", "i8_oracle.c", "i8_oracle.h"):
        shutil.copy(os.path.join(ORACLE, f), os.path.join(pkg, f))
    path = os.path.join(pkg, fname)
    with open(path) as fh:
        src = fh.read()
    if planted:
        with open(path, "w") as fh:
            fh.write(_plant(src, anchor, old, new))
    import oracle
    cc = subprocess.run(["gcc", *oracle.CFLAGS, os.path.join(pkg, "i8_oracle.c"),
                         "-o", os.path.join(pkg, "liboracle.so"), "-lm"],
                        capture_output=True, text=True)
    if cc.returncode != 0:
        return "compile_error", cc.stderr[-2000:]
    env = dict(os.environ, I8_ORACLE_DIR=pkg, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", *PIN_FILES, "-x", "-q",
                        "-p", "no:cacheprovider", "-m", "not gpu"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    tail = (r.stdout + r.stderr)[-3000:]
    if r.returncode == 0:
        return "survived", tail
    last = r.stdout.strip().splitlines()[-1] if r.stdout.strip() else ""
    if r.returncode == 1 and "failed" in last:
        first = re.search(r"^FAILED (\S+)", r.stdout, re.M)
        return "killed", first.group(1) if first else tail
    return "other", tail


@pytest.fixture(scope="module")
def outcomes():
    import oracle
    oracle.build()
    with tempfile.TemporaryDirectory(prefix="orc_mut_") as d:
        workers = max(1, min(8, os.cpu_count() or 1))
        cases = MUTANTS + [CONTROL]
        with ThreadPoolExecutor(max_workers=workers) as ex:
            res = list(ex.map(lambda m: _run_mutant(m, d), cases))
    return {m[0]: r for m, r in zip(cases, res)}


def test_every_mutation_site_exists():
    """Each planted slip names text that is really in the oracle, once per
    anchor (so a later edit of the oracle cannot silently turn a case into a
    no-op)."""
    for mid, fname, anchor, old, new in MUTANTS:
        with open(os.path.join(ORACLE, fname)) as fh:
            src = fh.read()
        assert src.count(anchor) == 1, mid
        assert old in src[src.index(anchor):], mid
        assert _plant(src, anchor, old, new) != src, mid


def test_unmodified_copy_passes_every_pin(outcomes):
    outcome, tail = outcomes[CONTROL[0]]
    assert outcome == "survived", tail


@pytest.mark.parametrize("mid", [m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(outcomes, mid):
    outcome, tail = outcomes[mid]
    assert outcome == "killed", f"{mid}: {outcome}\n{tail}"
