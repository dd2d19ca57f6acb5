"""Seeded synthetic inputs for MoE expert-parallel dispatch/combine.

This package is shared by the CPU oracle's tests, the GPU parity tests and
the benchmark. It only draws random numbers and lays them out; it holds none
of the method's arithmetic (no routing, no quantisation, no reduction).
"""
from .workloads import (  # noqa: F401
    WORKLOADS,
    Workload,
    make_expert_outputs,
    make_indices,
    make_num_tokens,
    make_tokens,
    make_weights,
)
