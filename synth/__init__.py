"""Seeded synthetic inputs for the GDN ReplaySSM verify / accept / flush path.

This package holds no arithmetic of the method itself: it only draws the
tensors (checkpoint state, committed buffer, draft blocks, accepted counts)
that both the CPU oracle and the CUDA library consume.
"""
from .workloads import (  # noqa: F401
    WORKLOADS,
    Workload,
    draft_block,
    initial_layer,
    seed_for,
)
