"""The C-ABI library on the host (CPU only: no compute call reaches a GPU).

- libmoe_gb300.so builds, loads and exports every function include/moe_gb300.h
  declares;
- invalid arguments are rejected on the host, before any CUDA call, with the
  documented status codes.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def lib():
    import token_dispatch_grouped_softmax_gb300 as moe

    moe.build()
    return moe.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_grouped_gemm_gate_up_swiglu", "moe_grouped_gemm_down",
              "moe_unpermute_combine", "moe_unpermute_combine_bwd", "moe_route_bwd",
              "moe_grouped_gemm_down_bwd", "moe_grouped_gemm_gate_up_bwd", "moe_gather_dx"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), "libmoe_gb300.so does not export %s" % n


def test_gemm_pairs_modes(lib):
    """0 single CTAs, 1 pairs for the forward and dgrad GEMMs, 2 pairs for
    gate_up only, 3 gate_up and the weight-gradient GEMMs."""
    try:
        for mode in (0, 1, 2, 3):
            assert lib.moe_set_gemm_pairs(mode) == 0
        assert lib.moe_set_gemm_pairs(4) == INVALID
        assert lib.moe_set_gemm_pairs(-1) == INVALID
    finally:
        lib.moe_set_gemm_pairs(2)


def test_version_and_error_strings(lib):
    assert lib.moe_version() == 10000
    assert lib.moe_error_string(0) == b"ok"
    assert lib.moe_error_string(4) == b"device-side wait timed out"
    assert lib.moe_error_string(99) == b"unknown status"


P = ctypes.c_void_p
FAKE = P(0x10000)       # a 16-byte aligned non-null pointer; never dereferenced on these paths
MISALIGNED = P(0x10002)

INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 5


def test_route_validation(lib):
    S = ctypes.c_size_t
    # k > E
    assert lib.moe_route(FAKE, FAKE, None, 4, 64, 4, 5, FAKE, FAKE, FAKE, None, 0, None) == INVALID
    # null x
    assert lib.moe_route(None, FAKE, None, 4, 64, 4, 2, FAKE, FAKE, FAKE, None, 0, None) == INVALID
    # H not a multiple of 8
    assert lib.moe_route(FAKE, FAKE, None, 4, 60, 4, 2, FAKE, FAKE, FAKE, None, 0, None) == UNSUPPORTED
    # E too large
    assert lib.moe_route(FAKE, FAKE, None, 4, 64, 2048, 2, FAKE, FAKE, FAKE, None, 0, None) == UNSUPPORTED
    # misaligned x
    assert lib.moe_route(MISALIGNED, FAKE, None, 4, 64, 4, 2, FAKE, FAKE, FAKE, None, 0, None) == INVALID
    # no workspace
    assert lib.moe_route(FAKE, FAKE, None, 4, 64, 8, 2, FAKE, FAKE, None, None, 0, None) == WORKSPACE
    n = S(0)
    assert lib.moe_route_workspace_size(4096, 2048, 128, ctypes.byref(n)) == 0
    # fused tensor-core router (E % 16 == 0, E <= 256): the split weight (3*H*E bf16) only
    assert n.value >= 3 * 2048 * 128 * 2
    assert lib.moe_route(FAKE, FAKE, None, 4096, 2048, 128, 8, FAKE, FAKE, None, FAKE, n.value - 1,
                         None) == WORKSPACE
    # split-K tensor-core router (other E % 8 == 0): split weight + fp32 partials
    assert lib.moe_route_workspace_size(4096, 2048, 200, ctypes.byref(n)) == 0
    assert n.value >= 3 * 2048 * 200 * 2 + 4096 * 200 * 4
    assert lib.moe_route_workspace_size(4, 64, 7, ctypes.byref(n)) == 0 and n.value >= 4 * 7 * 4
    # T == 0 is a valid no-op
    assert lib.moe_route(None, None, None, 0, 64, 4, 2, None, None, None, None, 0, None) == 0


def test_route_presplit_validation(lib):
    """The router on a split of W_r made once: the shapes of the tensor-core
    path only, its own (smaller) workspace, and the same argument checks."""
    S = ctypes.c_size_t
    n = S(0)
    # fused cluster router (E % 16 == 0, 16 <= E <= 256): no workspace at all
    assert lib.moe_route_presplit_workspace_size(4096, 2048, 128, ctypes.byref(n)) == 0 and n.value == 0
    # split-K tensor-core router: the fp32 partial logits only (no split weight)
    assert lib.moe_route_presplit_workspace_size(4096, 2048, 200, ctypes.byref(n)) == 0
    full = S(0)
    assert lib.moe_route_workspace_size(4096, 2048, 200, ctypes.byref(full)) == 0
    assert 4096 * 200 * 4 <= n.value < full.value
    assert lib.moe_route_presplit(FAKE, FAKE, None, 4096, 2048, 200, 8, FAKE, FAKE, None, FAKE, n.value - 1,
                                  None) == WORKSPACE
    # CUDA-core shapes have no split: refused
    assert lib.moe_route_presplit_workspace_size(4, 64, 7, ctypes.byref(n)) == UNSUPPORTED
    assert lib.moe_route_presplit(FAKE, FAKE, None, 4, 64, 7, 2, FAKE, FAKE, None, None, 0, None) == UNSUPPORTED
    assert lib.moe_route_split_weight(FAKE, 60, 16, FAKE, None) == UNSUPPORTED
    assert lib.moe_route_split_weight(FAKE, 64, 12, FAKE, None) == UNSUPPORTED
    # argument checks as moe_route
    assert lib.moe_route_presplit(FAKE, FAKE, None, 4, 64, 16, 17, FAKE, FAKE, None, None, 0, None) == INVALID
    assert lib.moe_route_presplit(MISALIGNED, FAKE, None, 4, 64, 16, 2, FAKE, FAKE, None, None, 0, None) == INVALID
    assert lib.moe_route_split_weight(None, 64, 16, FAKE, None) == INVALID
    assert lib.moe_route_split_weight(FAKE, 64, 16, MISALIGNED, None) == INVALID
    # T == 0 is a valid no-op
    assert lib.moe_route_presplit(None, None, None, 0, 64, 16, 2, None, None, None, None, 0, None) == 0


def test_ep_validation(lib):
    """The expert-parallel calls: argument checks before anything is enqueued,
    and the host-side EPLB plan's limits."""
    S = ctypes.c_size_t
    n = S(0)
    assert lib.moe_sort_chunks_workspace_size(8, 16, ctypes.byref(n)) == 0 and n.value >= (2 * 128 + 1) * 4
    assert lib.moe_sort_chunks_workspace_size(0, 16, ctypes.byref(n)) == INVALID
    assert lib.moe_sort_chunks(FAKE, 8, 16, 10, FAKE, FAKE, FAKE, None, 0, None) == WORKSPACE
    assert lib.moe_sort_chunks(None, 8, 16, 10, FAKE, FAKE, FAKE, FAKE, 4096, None) == INVALID
    assert lib.moe_sort_chunks(FAKE, 8, 16, 10, None, FAKE, FAKE, FAKE, 4096, None) == INVALID
    assert lib.moe_sort_chunks(FAKE, 8, 16, -1, FAKE, FAKE, FAKE, FAKE, 4096, None) == INVALID
    assert lib.moe_ep_map_replicas(FAKE, 4, 2, 8, FAKE, FAKE, FAKE, 6, FAKE, None) == INVALID   # n_phys < E
    assert lib.moe_ep_map_replicas(None, 4, 2, 8, FAKE, FAKE, FAKE, 8, FAKE, None) == INVALID
    assert lib.moe_ep_map_replicas(None, 0, 2, 8, FAKE, FAKE, FAKE, 8, None, None) == 0        # empty batch
    import numpy as np
    load = np.array([5, 3, 0, 9], dtype=np.int64)
    out = [np.empty(8, np.int32), np.empty(4, np.int32), np.empty(4, np.int32), np.empty(8, np.int32)]
    ptr = lambda a: ctypes.c_void_p(a.ctypes.data)
    assert lib.moe_eplb_plan(ptr(load), 4, 3, 8, *map(ptr, out), None) == INVALID    # 8 % 3 != 0
    assert lib.moe_eplb_plan(ptr(load), 4, 2, 3, *map(ptr, out), None) == INVALID    # fewer slots than experts
    bad = np.array([5, -1, 0, 9], dtype=np.int64)
    assert lib.moe_eplb_plan(ptr(bad), 4, 2, 8, *map(ptr, out), None) == INVALID     # a negative load
    assert lib.moe_eplb_plan(ptr(load), 4, 2, 8, *map(ptr, out), None) == 0
    assert sorted(out[3].tolist()) == list(range(8))


def test_permute_validation(lib):
    n = ctypes.c_size_t(0)
    assert lib.moe_permute_workspace_size(100, 8, 128, ctypes.byref(n)) == 0 and n.value >= 128 * 4
    pm = lib.moe_permute
    assert pm(FAKE, None, 100, 8, 128, FAKE, FAKE, FAKE, FAKE, None, None, 0, None) == WORKSPACE
    assert pm(FAKE, None, 100, 8, 128, FAKE, FAKE, FAKE, FAKE, None, FAKE, 4, None) == WORKSPACE
    assert pm(FAKE, None, 100, 0, 128, FAKE, FAKE, FAKE, FAKE, None, FAKE, n.value, None) == INVALID
    assert pm(FAKE, None, 100, 8, 4096, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 30, None) == UNSUPPORTED
    assert pm(None, None, 100, 8, 128, FAKE, FAKE, FAKE, FAKE, None, FAKE, n.value, None) == INVALID
    # w and w_perm come together
    assert pm(FAKE, FAKE, 100, 8, 128, FAKE, FAKE, FAKE, FAKE, None, FAKE, n.value, None) == INVALID
    # the workspace holds the grid-barrier counters: 16-byte aligned
    assert pm(FAKE, None, 100, 8, 128, FAKE, FAKE, FAKE, FAKE, None, MISALIGNED, n.value, None) == INVALID


def test_permute_rows_validation(lib):
    """The row moves: gather (src_row) and scatter (row_map)."""
    g, sc = lib.moe_permute_rows, lib.moe_permute_rows_scatter
    assert g(FAKE, FAKE, 64, 60, FAKE, None) == UNSUPPORTED                 # H % 8
    assert g(None, FAKE, 64, 64, FAKE, None) == INVALID
    assert g(MISALIGNED, FAKE, 64, 64, FAKE, None) == INVALID
    assert g(None, None, 0, 64, None, None) == 0                            # no rows
    assert sc(FAKE, FAKE, 16, 33, 64, FAKE, None) == UNSUPPORTED            # k > 32
    assert sc(FAKE, FAKE, 16, 2, 60, FAKE, None) == UNSUPPORTED             # H % 8
    assert sc(FAKE, FAKE, 16, 0, 64, FAKE, None) == INVALID
    assert sc(FAKE, None, 16, 2, 64, FAKE, None) == INVALID
    assert sc(FAKE, FAKE, 16, 2, 64, MISALIGNED, None) == INVALID
    assert sc(FAKE, FAKE, 1 << 30, 8, 64, FAKE, None) == INVALID            # T*k past int32
    assert sc(None, None, 0, 2, 64, None, None) == 0                        # an empty batch


def test_gemm_validation(lib):
    f = lib.moe_grouped_gemm_gate_up_swiglu
    # H not a multiple of 64
    assert f(FAKE, FAKE, FAKE, FAKE, 64, 128, 96, 8, 64, FAKE, None, None, None, None) == UNSUPPORTED
    # I not a multiple of 64
    assert f(FAKE, FAKE, FAKE, FAKE, 64, 128, 128, 8, 96, FAKE, None, None, None, None) == UNSUPPORTED
    # dense mode (no offsets) needs E == 1
    assert f(FAKE, None, None, FAKE, 128, 128, 128, 8, 64, FAKE, None, None, None, None) == INVALID
    # rows in order (no src_row) need T >= R
    assert f(FAKE, None, None, FAKE, 64, 128, 128, 1, 64, FAKE, None, None, None, None) == INVALID
    # h_w needs the permuted gate weights
    assert f(FAKE, FAKE, FAKE, FAKE, 64, 128, 128, 8, 64, FAKE, None, FAKE, FAKE, None) == INVALID
    # misaligned output
    assert f(FAKE, FAKE, FAKE, FAKE, 64, 128, 128, 8, 64, MISALIGNED, None, None, None, None) == INVALID
    # R == 0 is a valid no-op
    assert f(None, None, FAKE, None, 0, 0, 128, 8, 64, None, None, None, None, None) == 0
    g = lib.moe_grouped_gemm_down
    assert g(FAKE, FAKE, FAKE, 128, 100, 8, 64, FAKE, None) == UNSUPPORTED
    assert g(None, FAKE, FAKE, 128, 128, 8, 64, FAKE, None) == INVALID
    b1 = lib.moe_grouped_gemm_down_bwd
    assert b1(FAKE, FAKE, None, FAKE, FAKE, FAKE, 128, 128, 8, 64, FAKE, FAKE, FAKE, None) == INVALID
    assert b1(FAKE, FAKE, FAKE, None, FAKE, FAKE, 128, 128, 8, 64, FAKE, FAKE, FAKE, None) == INVALID
    assert b1(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 128, 8, 64, FAKE, FAKE, None, None) == INVALID
    n = ctypes.c_int64(0)
    assert lib.moe_grouped_gemm_down_bwd_parts(768, ctypes.byref(n)) == 0 and n.value == 12
    b2 = lib.moe_grouped_gemm_gate_up_bwd
    assert b2(FAKE, FAKE, FAKE, FAKE, FAKE, 64, 128, 128, 8, 64, FAKE, None, None) == INVALID


def test_combine_and_backward_validation(lib):
    assert lib.moe_unpermute_combine(FAKE, FAKE, FAKE, None, 4, 64, 33, FAKE, None) == UNSUPPORTED
    assert lib.moe_unpermute_combine(FAKE, FAKE, FAKE, None, 4, 60, 2, FAKE, None) == UNSUPPORTED
    assert lib.moe_unpermute_combine(FAKE, None, FAKE, None, 4, 64, 2, FAKE, None) == INVALID
    assert lib.moe_unpermute_combine(FAKE, FAKE, FAKE, MISALIGNED, 4, 64, 2, FAKE, None) == INVALID
    assert lib.moe_unpermute_combine_bwd(FAKE, None, 4, 64, 2, FAKE, None) == INVALID
    assert lib.moe_unpermute_combine_bwd(FAKE, FAKE, 4, 60, 2, FAKE, None) == UNSUPPORTED
    assert lib.moe_route_bwd(FAKE, 3, FAKE, FAKE, FAKE, 4, 2, 3, FAKE, None, None) == INVALID
    assert lib.moe_route_bwd(FAKE, 0, FAKE, FAKE, FAKE, 4, 8, 3, FAKE, None, None) == INVALID
    n = ctypes.c_size_t(0)
    assert lib.moe_gather_dx_workspace_size(64, 8, ctypes.byref(n)) == 0 and n.value == 64 * 8 * 4
    # the router term needs both d_logits and w_router, and the workspace
    assert lib.moe_gather_dx(FAKE, FAKE, FAKE, FAKE, None, 4, 64, 8, 2, FAKE, FAKE, n.value, None) == INVALID
    assert lib.moe_gather_dx(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 8, 2, FAKE, None, 0, None) == WORKSPACE
    # an empty batch is a no-op whatever its row pointers (an empty tensor's data pointer is NULL)
    assert lib.moe_gather_dx(None, None, None, None, FAKE, 0, 64, 8, 2, None, None, 0, None) == 0
    assert lib.moe_route_bwd_weight(FAKE, FAKE, 4, 64, 8, None, None) == INVALID


def test_python_binding_refuses_cpu_tensors():
    """The binding has no CPU fallback: CPU tensors are rejected."""
    import torch

    import token_dispatch_grouped_softmax_gb300 as moe

    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    wr = torch.zeros(64, 8, dtype=torch.float32)
    with pytest.raises(ValueError):
        moe.route(x, wr, 2)
