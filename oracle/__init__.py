"""CPU oracle for the Jacobi 5-point solver (test infrastructure only).

Only the test suite, the package smoke check and the benchmark's CPU
baseline / reference arm import this package.  The product path never does.
"""
from .oracle import (  # noqa: F401
    OracleInfo,
    h2,
    scale_source,
    sweep,
    residual,
    jacobi_run,
    rb_half_sweep,
    rb_run,
    axpy,
    task_sequence,
    barrier_stress_expected,
    has_openmp,
)
