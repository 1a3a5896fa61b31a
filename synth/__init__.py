"""Seeded synthetic inputs for the paged-attention hot path.

This package only draws random numbers and lays out the request batches; it
holds none of the method's arithmetic (no page addressing, no attention).  It is
the one module that both the CUDA path's tests/bench and the CPU oracle read.
"""
from .workloads import (  # noqa: F401
    SENTINEL_BF16,
    Request,
    Seq,
    Step,
    Workload,
    CONFIG_NAMES,
    EXTRA_NAMES,
    chunk_schedule,
    make_workload,
    make_prompt_workload,
    make_random_workload,
    make_prefix_groups_workload,
    make_shared_prefix_workload,
    make_tree_workload,
    random_tree,
    tree_mask_rows,
)
