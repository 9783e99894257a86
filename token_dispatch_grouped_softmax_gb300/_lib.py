"""ctypes loader of libmoe_gb300.so and its C signatures (include/moe_gb300.h).

There is no fallback: if the library is missing or fails to load, every call
raises.  Build it with ``token_dispatch_grouped_softmax_gb300.build()`` (or
``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes
import os

from . import _build

P = ctypes.c_void_p
I64 = ctypes.c_int64
SZ = ctypes.c_size_t
INT = ctypes.c_int

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
                4: "MOE_ERR_TIMEOUT", 5: "MOE_ERR_WORKSPACE", 6: "MOE_ERR_DEVICE",
                7: "MOE_ERR_SCRATCH_LIMIT"}

# name -> argtypes (every entry point returns int)
SIGNATURES = {
    "moe_version": [],
    "moe_sync_status": [P, ctypes.POINTER(ctypes.c_uint32)],
    "moe_set_wait_limit_ns": [ctypes.c_uint64],
    "moe_test_stall_gemm_producer": [INT],
    "moe_set_gemm_pairs": [INT],
    "moe_set_pdl": [INT],
    "moe_route_workspace_size": [I64, I64, I64, ctypes.POINTER(SZ)],
    "moe_route": [P, P, P, I64, I64, I64, I64, P, P, P, P, SZ, P],
    "moe_route_split_weight": [P, I64, I64, P, P],
    "moe_route_presplit_workspace_size": [I64, I64, I64, ctypes.POINTER(SZ)],
    "moe_route_presplit": [P, P, P, I64, I64, I64, I64, P, P, P, P, SZ, P],
    "moe_permute_workspace_size": [I64, I64, I64, ctypes.POINTER(SZ)],
    "moe_permute": [P, P, I64, I64, I64, P, P, P, P, P, P, SZ, P],
    "moe_permute_noalloc": [P, P, I64, I64, I64, P, P, P, P, P, P],
    "moe_permute_rows": [P, P, I64, I64, P, P],
    "moe_permute_rows_scatter": [P, P, I64, I64, I64, P, P],
    "moe_grouped_gemm_gate_up_swiglu": [P, P, P, P, I64, I64, I64, I64, I64, P, P, P, P, P],
    "moe_grouped_gemm_down": [P, P, P, I64, I64, I64, I64, P, P],
    "moe_unpermute_combine": [P, P, P, P, I64, I64, I64, P, P],
    "moe_unpermute_combine_bwd": [P, P, I64, I64, I64, P, P],
    "moe_route_bwd": [P, I64, P, P, P, I64, I64, I64, P, P, P],
    "moe_grouped_gemm_down_bwd_parts": [I64, ctypes.POINTER(I64)],
    "moe_grouped_gemm_down_bwd": [P, P, P, P, P, P, I64, I64, I64, I64, P, P, P, P],
    "moe_grouped_gemm_gate_up_bwd": [P, P, P, P, P, I64, I64, I64, I64, I64, P, P, P],
    "moe_gather_dx_workspace_size": [I64, I64, ctypes.POINTER(SZ)],
    "moe_gather_dx": [P, P, P, P, P, I64, I64, I64, I64, P, P, SZ, P],
    "moe_route_bwd_weight": [P, P, I64, I64, I64, P, P],
    "moe_sort_chunks_workspace_size": [I64, I64, ctypes.POINTER(SZ)],
    "moe_sort_chunks": [P, I64, I64, I64, P, P, P, P, SZ, P],
    "moe_ep_map_replicas": [P, I64, I64, I64, P, P, P, I64, P, P],
    "moe_eplb_plan": [P, I64, I64, I64, P, P, P, P, P],
}

_lib = None


class MoEError(RuntimeError):
    def __init__(self, name, status, detail=None):
        self.status = status
        msg = "%s failed: %s (%d)" % (name, STATUS_NAMES.get(status, "?"), status)
        if detail:
            msg += ", device status word 0x%08x" % detail
        super().__init__(msg)


def lib_path() -> str:
    return _build.LIB


def load():
    """The loaded library (raises when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError("libmoe_gb300.so is not built (%s); run "
                               "token_dispatch_grouped_softmax_gb300.build()" % _build.LIB)
        try:
            import torch  # noqa: F401  (loads the CUDA runtime the library shares)
        except ImportError:
            pass
        lib = ctypes.CDLL(_build.LIB)
        for name, argtypes in SIGNATURES.items():
            f = getattr(lib, name)
            f.argtypes = argtypes
            f.restype = INT
        lib.moe_error_string.argtypes = [INT]
        lib.moe_error_string.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def check(name, rc):
    if rc != MOE_OK:
        raise MoEError(name, rc)
    return rc


def call(name, *args):
    return check(name, getattr(load(), name)(*args))
