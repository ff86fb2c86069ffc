"""The oracle's pins catch planted mistakes.

Each case plants one plausible mistake in a copy of oracle/oracle.c (a swapped
nibble order, a wrong block-scale index, a dropped sign or term, a wrong
exponent bias, a transposed index ...), builds it on the CPU, and runs the pin
suite (tests/test_oracle_pins.py) against that build: the suite must fail.  A
control build of the unmodified source must pass.
"""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, text to find, replacement, which occurrence (0-based) or None for all)
MUTANTS = [
    ("nibble_order", "(k % 2 == 0) ? (byte & 0x0F) : (byte >> 4)",
     "(k % 2 == 0) ? (byte >> 4) : (byte & 0x0F)", None),
    ("nvfp4_scale_block", "scales[n * (K / 16) + k / 16]", "scales[n * (K / 16) + k / 32]", None),
    ("nvfp4_scale_row", "scales[n * (K / 16) + k / 16]", "scales[(n / 2) * (K / 16) + k / 16]", None),
    ("gscale_dropped", "* oracle_e4m3_to_f64(sc) * gscale;", "* oracle_e4m3_to_f64(sc);", None),
    ("e2m1_sign", "v = ldexp(1.0 + 0.5 * (double)m, e - 1);\n    return s ? -v : v;",
     "v = ldexp(1.0 + 0.5 * (double)m, e - 1);\n    return v;", None),
    ("e2m1_subnormal", "v = 0.5 * (double)m;", "v = (double)m;", None),
    ("e2m1_bias", "ldexp(1.0 + 0.5 * (double)m, e - 1)", "ldexp(1.0 + 0.5 * (double)m, e)", None),
    ("e4m3_bias", "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)", None),
    ("e4m3_subnormal", "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)", None),
    ("e4m3_nan", "if (e == 15 && m == 7)", "if (e == 15 && m == 8)", None),
    ("fp8_scale_transposed", "(n / 128) * kb + (k / 128)", "(k / 128) * kb + (n / 128)", None),
    ("fp8_code_index", "codes[n * K + k]", "codes[n * K + (k ^ 1)]", None),
    ("f16_subnormal", "ldexp((double)m, -24)", "ldexp((double)m, -25)", None),
    ("f16_bias", "ldexp(1.0 + (double)m / 1024.0, e - 15)", "ldexp(1.0 + (double)m / 1024.0, e - 14)", None),
    ("nvfp4_last_k_dropped", "for (int64_t k = 0; k < K; k++)", "for (int64_t k = 0; k < K - 1; k++)", 0),
    ("fp8_last_k_dropped", "for (int64_t k = 0; k < K; k++)", "for (int64_t k = 0; k < K - 1; k++)", 1),
    ("nvfp4_x_reversed", "oracle_f16_to_f64(x[m * K + k]) *\n                           nvfp4_weight",
     "oracle_f16_to_f64(x[m * K + (K - 1 - k)]) *\n                           nvfp4_weight", None),
    ("l1_without_abs", "mag += fabs(p);", "mag += p;", None),
    ("argmax_ties_high", "v > y[m * N + best]", "v >= y[m * N + best]", None),
    ("verify_count_off_by_one", "a = j + 1;", "a = j;", None),
    ("verify_bonus_index", "accept[1] = target[a];", "accept[1] = target[a > 0 ? a - 1 : 0];", None),
    ("verify_no_break", "            break;\n        a = j + 1;", "            continue;\n        a = j + 1;", None),
]


def _mutate(src, find, repl, occurrence):
    assert find in src, find
    if occurrence is None:
        return src.replace(find, repl)
    parts = src.split(find)
    assert len(parts) > occurrence + 1
    return find.join(parts[:occurrence + 1]) + repl + find.join(parts[occurrence + 1:])


def _run_pins(src_text, tmpdir, name):
    c = os.path.join(tmpdir, f"{name}.c")
    so = os.path.join(tmpdir, f"{name}.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", c, "-o", so, "-lm"])
    env = dict(os.environ, SKINNY_ORACLE_LIB=so, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return r.returncode, r.stdout[-2000:]


def test_pins_catch_every_planted_mistake():
    src = open(SRC).read()
    with tempfile.TemporaryDirectory() as td:
        jobs = [("control", src)] + [(n, _mutate(src, f, r, o)) for n, f, r, o in MUTANTS]
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            res = dict(zip([j[0] for j in jobs], ex.map(lambda j: _run_pins(j[1], td, j[0]), jobs)))
    rc, out = res.pop("control")
    assert rc == 0, "unmodified oracle must pass its pins:\n" + out
    survivors = [n for n, (rc, _) in res.items() if rc == 0]
    assert not survivors, f"planted mistakes not caught by any pin: {survivors}"
