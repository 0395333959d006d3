"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This package only draws numbers and lays them out (bit patterns, token ids, page
tables).  It contains none of the drafter's arithmetic.
"""
from .inputs import (  # noqa: F401
    DrafterConfig,
    Workload,
    CONFIGS,
    WORKLOADS,
    make_weights,
    make_workload,
    workload_taps,
)
