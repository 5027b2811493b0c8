"""Float64 CPU oracle for BDLM attention (test infrastructure only).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package. The CUDA library never does, and this package imports
nothing from it.
"""
from .bdlm_oracle import (  # noqa: F401
    NEG_INF,
    attend,
    attend_bwd,
    bdlm_attention,
    dense_bdlm_attention,
    full_mask,
    group_attention,
    group_positions,
    lse_merge,
    mask_rows,
    partial_attention,
    task_attention,
    task_attention_bwd,
    valid_pairs,
)
