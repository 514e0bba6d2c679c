"""CPU oracle for the dense GEMM with a pointwise epilogue.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg use it; the library's compute path never does.
See ``oracle_gemm.c`` for the definition it implements and the passages it
follows.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(full decode tables against a second decode, closed forms, invariants, exact
rational brute force, hand-worked examples under ``tests/golden/``), and
``tests/test_oracle_mutants.py`` shows that planted mistakes fail those pins.
"""

from .oracle import (  # noqa: F401
    EPI_KINDS,
    apply_epi,
    Oracle,
    build,
    compile_source,
    decode,
    decode_scale,
    default,
    gemm,
    gemm_entries,
    gemm_epi,
    gemm_mx,
    host_threads,
    library_path,
    round_output,
)
