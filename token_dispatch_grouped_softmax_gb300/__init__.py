"""GB300-native MoE expert layer: top-k softmax routing, token permutation,
grouped SwiGLU expert GEMMs on the tcgen05 tensor cores, gate-weighted
combine, and their backward, in libmoe_gb300.so (hand-written sm_103a CUDA
behind a C ABI, include/moe_gb300.h).

This package is the thin Python binding: it marshals torch tensors (device
memory, streams) into the C entry points.  Nothing here computes the layer.
"""
from ._build import build, up_to_date
from ._lib import MoEError, lib_path, load
from .ops import (GEMM_PAIRS_ALL, GEMM_PAIRS_GATE_UP, GEMM_PAIRS_GATE_UP_WGRAD, GEMM_PAIRS_NONE, gather_dx, grouped_gemm_down,
                  grouped_gemm_down_bwd, grouped_gemm_gate_up_bwd, grouped_gemm_gate_up_swiglu, permute,
                  permute_rows, permute_rows_scatter, route, route_bwd, route_bwd_weight, route_split_weight, route_supports_split, set_gemm_pairs, set_pdl, set_wait_limit_ns,
                  sync_status, unpermute_combine, unpermute_combine_bwd)
from . import ep
from .ops import ep_map_replicas, eplb_plan, sort_chunks
from .layer import (ForwardGraph, ForwardState, MoELayer, MoELayerFunction, OverlappedForward,
                    PipelinedForward, moe_backward, moe_forward)

__all__ = [
    "build", "up_to_date", "MoEError", "lib_path", "load",
    "route", "route_split_weight", "route_supports_split", "permute", "permute_rows", "permute_rows_scatter", "grouped_gemm_gate_up_swiglu", "grouped_gemm_down",
    "unpermute_combine", "unpermute_combine_bwd", "route_bwd", "grouped_gemm_down_bwd",
    "grouped_gemm_gate_up_bwd", "gather_dx", "route_bwd_weight", "sync_status", "set_wait_limit_ns", "set_gemm_pairs",
    "GEMM_PAIRS_NONE", "GEMM_PAIRS_ALL", "GEMM_PAIRS_GATE_UP", "GEMM_PAIRS_GATE_UP_WGRAD",
    "set_pdl", "sort_chunks", "ep_map_replicas", "eplb_plan", "ep",
    "ForwardGraph", "ForwardState", "MoELayer", "OverlappedForward", "MoELayerFunction", "PipelinedForward", "moe_forward", "moe_backward",
]
