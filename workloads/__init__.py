"""Seeded synthetic inputs for the HSQ compressed-KV path.

This package draws random numbers and arranges them into arrays; it holds no
step of the method itself (no rotation, quantiser, RoPE, routing or
attention).  Both the float64 oracle and the CUDA library consume the arrays
it returns.  The one input that needs a method step to build -- the planted
needle, whose keys must line up with the query after rotary embedding --
takes the rotary function as an argument from its caller.
"""

from .configs import WORKLOADS, Workload, get_workload
from .generate import (
    LayerInputs,
    layer_inputs,
    layer_meta,
    qjl_matrix,
    queries,
    needle_groups,
    plant_needle,
    to_bf16_bits,
    round_to_bf16,
)

__all__ = [
    "WORKLOADS",
    "Workload",
    "get_workload",
    "LayerInputs",
    "layer_inputs",
    "layer_meta",
    "qjl_matrix",
    "queries",
    "needle_groups",
    "plant_needle",
    "to_bf16_bits",
    "round_to_bf16",
]
