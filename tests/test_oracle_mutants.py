"""Plausible mistakes planted in a copy of the oracle (on the CPU) must each
fail at least one of the pins in oracle_checks.py.  The real oracle source is
never modified; each mutant is compiled from a patched temporary copy."""
import os
import tempfile

import pytest

import oracle
from oracle import build as obuild
import oracle_checks as oc

MUTANTS = {
    "nibble_order_swapped": ("(k & 1) ? (unsigned)(b >> 4) : (unsigned)(b & 15u)",
                             "(k & 1) ? (unsigned)(b & 15u) : (unsigned)(b >> 4)"),
    "scale_block_32": ("scales[n * (K / 16) + k / 16]", "scales[n * (K / 16) + k / 32]"),
    "scale_row_stride": ("scales[n * (K / 16) + k / 16]", "scales[n * (K / 32) + k / 16]"),
    "code_row_stride": ("codes[n * (K / 2) + k / 2]", "codes[n * (K / 4) + k / 2]"),
    "global_scale_dropped": ("return v * s * (double)gs;", "return v * s;"),
    "e2m1_bias": ("ldexp(1.0 + (double)m / 2.0, (int)e - 1)", "ldexp(1.0 + (double)m / 2.0, (int)e)"),
    "e2m1_subnormal": ("mag = ldexp((double)m, -1);", "mag = ldexp((double)m, 0);"),
    "e2m1_sign_dropped": ("  return s ? -mag : mag;\n}\n\n/* E4M3", "  return mag;\n}\n\n/* E4M3"),
    "e4m3_bias": ("ldexp(1.0 + (double)m / 8.0, (int)e - 7)", "ldexp(1.0 + (double)m / 8.0, (int)e - 8)"),
    "e4m3_subnormal": ("ldexp((double)m / 8.0, 1 - 7)", "ldexp((double)m / 8.0, -7)"),
    "e4m3_nan_missing": ("if (e == 15u && m == 7u) return NAN;", ""),
    "bf16_mantissa": ("(double)m / 128.0, (int)e - 127", "(double)m / 256.0, (int)e - 127"),
    "x_k_reversed": ("nvfp4_oracle_bf16(x[m * K + k])", "nvfp4_oracle_bf16(x[m * K + (K - 1 - k)])"),
    "output_transposed": ("&y[m * N + n], &absdot[m * N + n]", "&y[n * M + m], &absdot[n * M + m]"),
    "absdot_signed": ("aacc += fabs(t);", "aacc += t;"),
    "first_term_dropped": ("for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 1; k < K; ++k) {"),
}


@pytest.fixture(scope="module")
def source():
    with open(obuild.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, "mutation anchor must match exactly once: %r" % old
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    lib = obuild.compile_source(str(src), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for check in oc.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, "no pin catches mutant %s" % name
