"""Planted mistakes: each test copies the oracle's C source, plants one
plausible error, compiles the copy, and runs the pin suite against it.  The
pins must catch every one of them (the suite must fail)."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mxfp4_oracle.c")

MUTANTS = {
    "amax_rounding_constant": ("u = (u + 0x200000u) & 0xFF800000u;", "u = (u + 0x400000u) & 0xFF800000u;"),
    "scale_exponent_offset": ("int s = e - 129;", "int s = e - 128;"),
    "ties_to_odd": ("(c & 1) == 0 && (best & 1) == 1", "(c & 1) == 1 && (best & 1) == 0"),
    "saturate_to_code_6": ("uint8_t best = 7;", "uint8_t best = 6;"),
    "odd_index_in_low_nibble": ("(uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4))",
                                "(uint8_t)(codes[2 * i + 1] | (codes[2 * i] << 4))"),
    "negative_zero_loses_sign": ("int neg = signbit(q) ? 1 : 0;", "int neg = (q < 0) ? 1 : 0;"),
    "gemm_drops_b_scale": ("double vb = oracle_e2m1_decode(bc) * oracle_e8m0_decode(bs[n * nblk + k / 32]);",
                           "double vb = oracle_e2m1_decode(bc);"),
    "gemm_transposed_operand": ("uint8_t ab = aq[m * kh + k / 2], bb = bq[n * kh + k / 2];",
                                "uint8_t ab = aq[m * kh + k / 2], bb = bq[(n % M) * kh + k / 2];"),
    "bf16_truncates": ("r = ldexp(nearbyint(ldexp(d, -quantum)), quantum);",
                       "r = ldexp(trunc(ldexp(d, -quantum)), quantum);"),
    "e8m0_bias_off_by_one": ("return ldexp(1.0, (int)byte - 127);", "return ldexp(1.0, (int)byte - 126);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle.compile_source(str(src), str(tmp_path / "libmutant.so"))
    env = dict(os.environ, MXFP4_ORACLE_VARIANT_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0 and "failed" in r.stdout, f"pins did not catch '{name}':\n{r.stdout[-2000:]}"
