"""CPU oracle for the ternary (PQ2) x INT8 matmul — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA library: the
arithmetic lives in ``pq2_oracle.c`` (plain C, IEEE fp32/fp64, no FMA
contraction), and this module only marshals numpy arrays into it.
"""
from .oracle import (  # noqa: F401
    build_oracle,
    decode_field,
    half_to_float,
    bf16_to_float,
    float_to_bf16_rne,
    prepare,
    decode_matrix,
    widen,
    quantize,
    q_planes,
    qsum,
    group_dots,
    scale_accumulate,
    linear,
    within_bound,
    bf16_within_bound,
)
