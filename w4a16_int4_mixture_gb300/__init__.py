"""GB300 (sm_103a) W4A16 INT4 Mixture-of-Experts expert computation.

BF16 activations x INT4 weights with group-32 BF16 scales: moe_align routing,
gate/up GEMM with a fused SiLU(gate)*up epilogue, down GEMM and the top-k
weighted combine, as hand-written tcgen05/TMA kernels behind a C ABI
(include/chord.h).  This package holds the in-tree build of that library and a
thin PyTorch-facing binding; it has no CPU implementation of the path.
"""

from ._build import build  # noqa: F401
from .ops import (  # noqa: F401
    ChordError,
    describe_schedule,
    get_device_error,
    grouped_workspace_size,
    moe_align,
    moe_align_capacity,
    moe_route_align,
    moe_workspace_size,
    PackedWeights,
    prepack,
    prepack_size,
    prepack_weights,
    select_block_m,
    stage_timing_enable,
    stage_timing_read,
    w4a16_moe,
    w4a16_moe_grouped,
    w4a16_moe_indexed,
)
from . import synth  # noqa: F401

__all__ = [
    "build", "ChordError", "describe_schedule", "get_device_error", "grouped_workspace_size",
    "moe_align", "moe_align_capacity", "moe_route_align", "moe_workspace_size", "PackedWeights",
    "prepack", "prepack_size", "prepack_weights", "select_block_m",
    "stage_timing_enable", "stage_timing_read", "w4a16_moe", "w4a16_moe_grouped",
    "w4a16_moe_indexed", "synth",
]
