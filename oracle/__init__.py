"""CPU oracle for the skinny weight-only linear layer (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never does, and this package imports nothing from it.

Parity status of every function here: pinned (see ``tests/test_oracle_pins.py``).
"""
from .oracle import (  # noqa: F401
    build,
    f16_to_f64,
    e2m1_to_f64,
    e4m3_to_f64,
    nvfp4_linear,
    fp8_linear,
    argmax_rows,
    verify,
    tolerance,
    threads,
    set_threads,
)
from .quant import e2m1_round, e4m3_round, quantize_fp8, quantize_nvfp4  # noqa: F401
from .sample import margin as sample_margin, sample, sample_row  # noqa: F401
