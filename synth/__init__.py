"""Seeded synthetic inputs shared by the CUDA path's tests, the oracle's tests and the bench.

This package draws random numbers and nothing else: fp32 weight matrices, the
rows that carry salient input channels, act-order group maps and activation
matrices.  It holds none of the quantization or product arithmetic; that lives
on each side of the parity check separately.
"""

from .inputs import (  # noqa: F401
    WORKLOADS,
    Workload,
    activations,
    act_order_g_idx,
    gaussian_weights,
    salient_rows,
    student_t_weights,
    weights_for,
)
