"""Seeded synthetic inputs for the sparse-delta-memory forward (Phase 1 + decay-and-write) and
the backward's Phase A, GWR and GDS, and the forward's read-side gather.

This package is shared by the tests, the benchmark and the oracle's callers. It only draws
random numbers and lays them out; it holds none of the method's arithmetic.
"""

from .workloads import (  # noqa: F401
    WORKLOADS,
    Workload,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    make_backward_inputs,
    make_bank_stream,
    make_grad_stream,
    make_snapshot_chunk,
    make_inputs,
    make_read_grads,
    make_read_weights,
    make_write_weights,
    scaled,
)
