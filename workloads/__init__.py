"""Seeded synthetic inputs for block-sparse routed attention.

This module only draws random numbers and rounds them to BF16.  It holds none
of the method's arithmetic: no pooling, routing, selection or attention.  Both
the CUDA path (through tests and the benchmark) and the CPU oracle consume the
arrays it returns.
"""

from .synth import (  # noqa: F401
    REWEIGHT_WORKLOADS,
    WORKLOADS,
    Workload,
    bf16_round_bits,
    make_anchors,
    make_inputs,
    make_reweight_workload,
    make_workload,
)
