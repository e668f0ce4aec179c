"""Plant plausible mistakes in a copy of the oracle and show the pins catch each.

Every mutant below is a one-token change of the kind that slips into such code
(a dropped term, a wrong sign, a transposed index, an off-by-one).  The copy is
compiled into a temporary directory on the CPU; the committed oracle is never
touched.  For each mutant at least one pin must fail.
"""
import os
import shutil

import pytest

import oracle
import oracle_pins

SRC = oracle.SOURCE

MUTANTS = {
    "bias dropped": ("return s + (bias ? (double)bias[j] : 0.0);", "return s;"),
    "B read transposed": ("in_value(B, dtype, t * N + j)", "in_value(B, dtype, j * K + t)"),
    "K loop short by one": ("for (int64_t t = 0; t < K; ++t)", "for (int64_t t = 0; t + 1 < K; ++t)"),
    "leaky slope sign": ("z > 0.0 ? z : alpha * z", "z > 0.0 ? z : -alpha * z"),
    "relu passes negatives": ("z > 0.0 ? z : 0.0", "z > 0.0 ? z : 0.5 * z"),
    "tanh numerator sign": ("(ep - em) / (ep + em)", "(em - ep) / (ep + em)"),
    "tanh saturation wrong": ("if (z > 20.0) return 1.0;", "if (z > 2.0) return 1.0;"),
    "sigmoid exponent sign": ("return 1.0 / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(z));"),
    "gelu erf scale": ("erf(z / sqrt(2.0))", "erf(z / 2.0)"),
    "gelu half dropped": ("return 0.5 * z * (1.0 + erf", "return z * (1.0 + erf"),
    "conv dilation dropped (rows)": ("r * g->dh", "r"),
    "conv dilation dropped (cols)": ("q * g->dw", "q"),
    "conv pad sign": ("oh * g->sh - g->pt", "oh * g->sh + g->pt"),
    "conv stride axes swapped": ("ow * g->sw", "ow * g->sh"),
    "conv left pad used for top": ("oh * g->sh - g->pt", "oh * g->sh - g->pl"),
    "conv filter taps transposed": ("((co * g->C + ci) * g->kh + r) * g->kw + q",
                                    "((co * g->C + ci) * g->kh + q) * g->kw + r"),
    "conv bias per channel lost": ("(double)bias[co]", "(double)bias[0]"),
    "conv out-dim off by one": ("dil * (k - 1) - 1;", "dil * (k - 1);"),
    "conv skips padding check": ("if (ih < 0 || ih >= g->H || iw < 0 || iw >= g->W) continue;",
                                 "if (ih < 0 || iw < 0) continue;"),
    "residual dropped": ("return R ? z + residual_value(R, rdtype, idx) : z;", "return z;"),
    "residual after the activation": ("oracle_act(add_residual(z, R, rdtype, idx), act, alpha)",
                                      "add_residual(oracle_act(z, act, alpha), R, rdtype, idx)"),
    "residual codes read as bf16": ("return in_value(R, rdtype, idx);", "return in_value(R, OR_BF16, idx);"),
    "fp32 inputs narrowed": ("if (dtype == OR_F32) return (double)((const float *)p)[idx];",
                             "if (dtype == OR_F32) return (double)(_Float16)((const float *)p)[idx];"),
    "f16 exponent bias": ("e - 15)", "e - 14)"),
    "f16 subnormal scale": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "bf16 fraction width": ("(double)f / 128.0", "(double)f / 256.0"),
    "bf16 exponent bias": ("e - 127)", "e - 126)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation anchor not found: {old!r}"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle.build(str(src), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib, str(src))
    failures = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, ValueError):
            failures.append(check.__name__)
    assert failures, f"no pin caught the mutant '{name}'"
