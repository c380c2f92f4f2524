"""fp64 CPU oracle for streaming Nystrom (landmark) attention.

Test infrastructure only: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` are its only users.  The product path never
imports it.
"""
from .nystrom_oracle import (  # noqa: F401
    AGGREGATE, FM, DEN_EPS, EXACT_SLACK, RIDGE_REL, RIDGE_TRIES,
    DEFAULT_M, DEFAULT_W, DEFAULT_SINK,
    NystromOracle, RidgeResult, StepDiag, cholesky_lower, direct_output,
    effective_landmarks, f32_round, is_exact_only, ridge_pinv, score_scale,
    seg_means,
)
