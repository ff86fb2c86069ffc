"""The pins of the quantizer and sampler oracles catch planted mistakes.

Each case plants one plausible mistake in a copy of oracle/quant.py or
oracle/sample.py (a wrong format maximum or scale divisor, ties rounded away
from even, the sign of zero lost, the nibble order swapped, the zero-scale
case dropped, ties in the candidate order broken the wrong way, the top-p cut
one short, the temperature applied the wrong way round, one candidate too
many, the draw scaled by the wrong total), and
runs the pin suites (tests/test_oracle_quant.py, tests/test_oracle_sample.py)
against that copy: they must fail.  A control copy must pass.
"""
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, file in oracle/, text to find, replacement)
MUTANTS = [
    ("fp8_format_max", "quant.py", "_F32(a / _F32(448.0))", "_F32(a / _F32(240.0))"),
    ("fp8_zero_block_scale", "quant.py", "if a > 0 else _F32(1.0)", "if a > 0 else _F32(0.5)"),
    ("nvfp4_tensor_divisor", "quant.py", "_F32(A / _F32(2688.0))", "_F32(A / _F32(448.0))"),
    ("nvfp4_block_divisor", "quant.py", "(b / _F32(6.0))", "(b / _F32(4.0))"),
    ("ties_away_from_even", "quant.py",
     "((d_hi == d_lo) & ((codes[hi] & 1) == 0) & ((codes[lo] & 1) == 1))", "(d_hi == d_lo)"),
    ("zero_sign_lost", "quant.py", "np.where(np.signbit(v), out | sign_bit, out)", "np.where(v < 0, out | sign_bit, out)"),
    ("nibble_order", "quant.py", "(nib[:, 0::2] | (nib[:, 1::2] << 4))", "(nib[:, 1::2] | (nib[:, 0::2] << 4))"),
    ("zero_scale_codes", "quant.py", "np.where(zero, np.where(np.signbit(blocks), 0x8, 0x0), nib)", "nib"),
    ("ties_high_index", "sample.py", "np.lexsort((np.arange(z.size), -z.astype(np.float64)))",
     "np.lexsort((-np.arange(z.size), -z.astype(np.float64)))"),
    ("top_p_one_short", "sample.py",
     'keep = int(np.searchsorted(cum, float(np.float32(top_p)) * cum[-1], side="left")) + 1',
     'keep = int(np.searchsorted(cum, float(np.float32(top_p)) * cum[-1], side="left"))'),
    ("temperature_inverted", "sample.py",
     "p = np.exp((zz - zz[0]) / float(np.float32(temperature)))\n    cum = np.cumsum(p)\n    keep",
     "p = np.exp((zz - zz[0]) * float(np.float32(temperature)))\n    cum = np.cumsum(p)\n    keep"),
    ("one_candidate_too_many", "sample.py", "order = _order(z)[:top_k]\n    if temperature <= 0:\n        return int",
     "order = _order(z)[:top_k + 1]\n    if temperature <= 0:\n        return int"),
    ("draw_over_all_candidates", "sample.py", "target = float(np.float32(u)) * cum[keep - 1]\n    j",
     "target = float(np.float32(u)) * cum[-1]\n    j"),
]

CONFTEST = '''import os
import sys

HERE = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU")
'''


def _run(name, file, find, repl, lib):
    td = tempfile.mkdtemp(prefix=f"mut_{name}_")
    try:
        shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(td, "oracle"),
                        ignore=shutil.ignore_patterns("_build", "__pycache__", "*.so"))
        shutil.copytree(os.path.join(ROOT, "synth"), os.path.join(td, "synth"),
                        ignore=shutil.ignore_patterns("__pycache__"))
        os.makedirs(os.path.join(td, "tests"))
        for t in ("test_oracle_quant.py", "test_oracle_sample.py"):
            shutil.copy(os.path.join(ROOT, "tests", t), os.path.join(td, "tests", t))
        with open(os.path.join(td, "tests", "conftest.py"), "w") as f:
            f.write(CONFTEST)
        if file:
            p = os.path.join(td, "oracle", file)
            src = open(p).read()
            assert src.count(find) == 1, (name, find)
            with open(p, "w") as f:
                f.write(src.replace(find, repl))
        env = dict(os.environ, SKINNY_ORACLE_LIB=lib, OMP_NUM_THREADS="1")
        r = subprocess.run([sys.executable, "-m", "pytest", "tests", "-x", "-q", "-p", "no:cacheprovider"],
                           cwd=td, env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        return r.returncode, r.stdout[-2000:]
    finally:
        shutil.rmtree(td, ignore_errors=True)


def test_pins_catch_every_planted_mistake_in_the_quantizer_and_sampler_oracles():
    pytest.importorskip("torch")
    import oracle

    lib = oracle.build()
    jobs = [("control", None, None, None)] + MUTANTS
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        res = dict(zip([j[0] for j in jobs], ex.map(lambda j: _run(j[0], j[1], j[2], j[3], lib), jobs)))
    rc, out = res.pop("control")
    assert rc == 0, "unmodified oracle must pass its pins:\n" + out
    survivors = [n for n, (rc, _) in res.items() if rc == 0]
    assert not survivors, f"planted mistakes not caught by any pin: {survivors}"
