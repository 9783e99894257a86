"""Per-step entry points of the MoE layer on torch CUDA tensors.

Argument marshalling only: each function checks dtypes and shapes, allocates
its outputs with torch (device memory), and calls the matching C entry point
of libmoe_gb300.so on the current torch stream.  Every step runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import call

_BF16 = torch.bfloat16


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (the path runs only on the GPU)" % name)
    if t.device.index != torch.cuda.current_device():
        # the kernels run on the current device and would be handed another GPU's memory
        raise ValueError("%s is on %s but the current device is cuda:%d" % (name, t.device,
                                                                           torch.cuda.current_device()))
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims" % (name, ndim))
    return t


def _ws(nbytes, device):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def sync_status():
    """Synchronise the current stream and raise if a kernel reported a device-side error."""
    detail = ctypes.c_uint32(0)
    call("moe_sync_status", _stream(), ctypes.byref(detail))
    return detail.value


def set_wait_limit_ns(ns: int):
    call("moe_set_wait_limit_ns", int(ns))


GEMM_PAIRS_NONE, GEMM_PAIRS_ALL, GEMM_PAIRS_GATE_UP, GEMM_PAIRS_GATE_UP_WGRAD = 0, 1, 2, 3


def set_gemm_pairs(mode):
    """Where the grouped GEMMs run: False / GEMM_PAIRS_NONE on single CTAs,
    True / GEMM_PAIRS_ALL every forward and dgrad GEMM on CTA pairs (2-SM
    MMAs), GEMM_PAIRS_GATE_UP the forward gate_up GEMM on pairs,
    GEMM_PAIRS_GATE_UP_WGRAD that and the two weight-gradient GEMMs.  The
    results are bit-identical."""
    call("moe_set_gemm_pairs", int(mode))


_pdl_on = [True]


def set_pdl(on: bool):
    """Programmatic dependent launch of every kernel (default on): a kernel's
    set-up overlaps the tail of the one before it on the stream.  Off for
    graphs whose kernels run beside another stream's (OverlappedForward)."""
    call("moe_set_pdl", 1 if on else 0)
    _pdl_on[0] = bool(on)


def pdl_enabled() -> bool:
    """The setting last made through set_pdl (the library starts with it on)."""
    return _pdl_on[0]


# ----------------------------------------------------------------- forward

def route(x, w_router, k, bias=None, return_logits=False, w_split=None):
    """ids [T,k] int32, w [T,k] fp32 (and logits [T,E] fp32).

    w_split: W_r's bf16 split from route_split_weight(w_router), made once
    while W_r does not change (moe_route_presplit); the results are the same
    bit for bit."""
    _need(x, "x", _BF16, 2)
    _need(w_router, "w_router", torch.float32, 2)
    if bias is not None:
        _need(bias, "bias", torch.float32, 1)
    T, H = x.shape
    E = w_router.shape[1]
    dev = x.device
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev) if return_logits else None
    nbytes = ctypes.c_size_t(0)
    if w_split is not None:
        _need(w_split, "w_split", _BF16, 2)
        if tuple(w_split.shape) != (3 * H, E):
            raise ValueError("w_split must be [3H, E] (route_split_weight)")
        call("moe_route_presplit_workspace_size", T, H, E, ctypes.byref(nbytes))
        ws = _ws(nbytes.value, dev) if nbytes.value else None
        call("moe_route_presplit", _p(x), _p(w_split), _p(bias), T, H, E, k, _p(ids), _p(w), _p(logits), _p(ws),
             ws.numel() if ws is not None else 0, _stream())
        return (ids, w, logits) if return_logits else (ids, w)
    call("moe_route_workspace_size", T, H, E, ctypes.byref(nbytes))
    ws = _ws(nbytes.value, dev)
    call("moe_route", _p(x), _p(w_router), _p(bias), T, H, E, k, _p(ids), _p(w), _p(logits), _p(ws),
         ws.numel(), _stream())
    return (ids, w, logits) if return_logits else (ids, w)


def route_supports_split(H, E):
    """Whether the router runs on the tensor cores at this shape (E % 8 == 0,
    H % 64 == 0, E <= 1024), the shapes route_split_weight serves."""
    return E % 8 == 0 and H % 64 == 0 and E <= 1024


def route_split_weight(w_router, out=None):
    """W_r's exact three-term bf16 split [3H, E] (W0 rows, then W1, then W2),
    for route(..., w_split=...) while W_r does not change.  out: an existing
    [3H, E] bf16 tensor to refresh in place (e.g. one a captured graph reads)."""
    _need(w_router, "w_router", torch.float32, 2)
    H, E = w_router.shape
    w_split = torch.empty((3 * H, E), dtype=_BF16, device=w_router.device) if out is None else out
    _need(w_split, "w_split", _BF16, 2)
    if tuple(w_split.shape) != (3 * H, E):
        raise ValueError("w_split must be [3H, E]")
    call("moe_route_split_weight", _p(w_router), H, E, _p(w_split), _stream())
    return w_split


def permute(ids, E, w=None):
    """counts [E], offsets [E+1], row_map [R], src_row [R] (int32), and with w
    [T,k] fp32 also w_perm [R] fp32 (the gate weight of each permuted row)."""
    _need(ids, "ids", torch.int32, 2)
    if w is not None:
        _need(w, "w", torch.float32, 2)
    T, k = ids.shape
    dev = ids.device
    nbytes = ctypes.c_size_t(0)
    call("moe_permute_workspace_size", T, k, E, ctypes.byref(nbytes))
    ws = _ws(nbytes.value, dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    row_map = torch.empty(T * k, dtype=torch.int32, device=dev)
    src_row = torch.empty(T * k, dtype=torch.int32, device=dev)
    w_perm = torch.empty(T * k, dtype=torch.float32, device=dev) if w is not None else None
    call("moe_permute", _p(ids), _p(w), T, k, E, _p(counts), _p(offsets), _p(row_map), _p(src_row),
         _p(w_perm), _p(ws), ws.numel(), _stream())
    if w is not None:
        return counts, offsets, row_map, src_row, w_perm
    return counts, offsets, row_map, src_row


def permute_rows(x, src_row, out=None):
    """out[r] = x[src_row[r]] for every row r (bf16 rows of width H); out: an
    existing contiguous [R, H] bf16 tensor (or row slice) to write into."""
    _need(x, "x", _BF16, 2)
    _need(src_row, "src_row", torch.int32, 1)
    R, H = src_row.shape[0], x.shape[1]
    if out is None:
        out = torch.empty((R, H), dtype=_BF16, device=x.device)
    else:
        _need(out, "out", _BF16, 2)
        if tuple(out.shape) != (R, H):
            raise ValueError("out must be [R, H]")
    call("moe_permute_rows", _p(x), _p(src_row), R, H, _p(out), _stream())
    return out


def permute_rows_scatter(x, row_map, k):
    """x_perm [T*k, H] bf16 with x_perm[row_map[t*k + j]] = x[t]: the rows of
    permute_rows(x, src_row) for the same permutation, moved token by token
    (each token row read once)."""
    _need(x, "x", _BF16, 2)
    _need(row_map, "row_map", torch.int32, 1)
    T, H = x.shape
    if row_map.shape[0] != T * k:
        raise ValueError("row_map must hold T*k entries")
    out = torch.empty((T * k, H), dtype=_BF16, device=x.device)
    call("moe_permute_rows_scatter", _p(x), _p(row_map), T, k, H, _p(out), _stream())
    return out


def sort_chunks(counts, N):
    """Rows arriving as an A x B chunk matrix in (a, b) order -> (b, a) order
    (moe_sort_chunks): src_of [N], pos_of [N] and group_offsets [B+1] (int32).
    counts: [A, B] int32 on the device, summing to N."""
    _need(counts, "counts", torch.int32, 2)
    A, B = counts.shape
    dev = counts.device
    src_of = torch.empty(N, dtype=torch.int32, device=dev)
    pos_of = torch.empty(N, dtype=torch.int32, device=dev)
    group = torch.empty(B + 1, dtype=torch.int32, device=dev)
    nbytes = ctypes.c_size_t(0)
    call("moe_sort_chunks_workspace_size", A, B, ctypes.byref(nbytes))
    ws = _ws(nbytes.value, dev)
    call("moe_sort_chunks", _p(counts), A, B, N, _p(src_of), _p(pos_of), _p(group), _p(ws), ws.numel(), _stream())
    return src_of, pos_of, group


def ep_map_replicas(ids, rep_first, rep_count, rep_list):
    """Logical expert ids [T, k] -> physical replica ids [T, k] (moe_ep_map_replicas);
    the plan tensors are int32 on the device."""
    _need(ids, "ids", torch.int32, 2)
    for t, n in ((rep_first, "rep_first"), (rep_count, "rep_count"), (rep_list, "rep_list")):
        _need(t, n, torch.int32, 1)
    T, k = ids.shape
    E, n_phys = rep_first.shape[0], rep_list.shape[0]
    out = torch.empty_like(ids)
    call("moe_ep_map_replicas", _p(ids), T, k, E, _p(rep_first), _p(rep_count), _p(rep_list), n_phys, _p(out),
         _stream())
    return out


def eplb_plan(expert_load, G, n_phys):
    """EPLB-style replication and placement on the host (moe_eplb_plan).
    expert_load: per-expert loads (sequence of ints); returns a dict of numpy
    arrays phys_to_log [n_phys], rep_first [E], rep_count [E], rep_list
    [n_phys] (int32) and rank_load [G] (int64)."""
    import numpy as np

    load = np.ascontiguousarray(np.asarray(expert_load, dtype=np.int64))
    E = load.shape[0]
    out = dict(phys_to_log=np.empty(n_phys, np.int32), rep_first=np.empty(E, np.int32),
               rep_count=np.empty(E, np.int32), rep_list=np.empty(n_phys, np.int32),
               rank_load=np.empty(G, np.int64))
    ptr = lambda a: ctypes.c_void_p(a.ctypes.data)
    call("moe_eplb_plan", ptr(load), E, G, n_phys, ptr(out["phys_to_log"]), ptr(out["rep_first"]),
         ptr(out["rep_count"]), ptr(out["rep_list"]), ptr(out["rank_load"]))
    return out


def grouped_gemm_gate_up_swiglu(x, src_row, offsets, gate_up, I, R=None, w_perm=None, save_for_backward=False):
    """h [R, I] bf16; with save_for_backward also gu_pre [R, 2I] fp32 and h_w = w_perm * h [R, I] bf16.
    src_row None: x is already in permuted order (or the dense mode when offsets is None too)."""
    _need(x, "x", _BF16, 2)
    _need(gate_up, "gate_up", _BF16, 2)
    T, H = x.shape
    E = gate_up.shape[0] // H
    if gate_up.shape != (E * H, 2 * I):
        raise ValueError("gate_up must be [E*H, 2I]")
    if src_row is not None:
        _need(src_row, "src_row", torch.int32, 1)
        R = src_row.shape[0]
    elif R is None:
        R = T
    if offsets is not None:
        _need(offsets, "offsets", torch.int32, 1)
    if w_perm is not None:
        _need(w_perm, "w_perm", torch.float32, 1)
    h = torch.empty((R, I), dtype=_BF16, device=x.device)
    gu = hw = None
    if save_for_backward:
        if w_perm is None:
            raise ValueError("save_for_backward needs w_perm (from permute(ids, E, w))")
        gu = torch.empty((R, 2 * I), dtype=torch.float32, device=x.device)
        hw = torch.empty((R, I), dtype=_BF16, device=x.device)
    call("moe_grouped_gemm_gate_up_swiglu", _p(x), _p(src_row), _p(offsets), _p(gate_up), T, R, H, E, I,
         _p(h), _p(w_perm), _p(gu), _p(hw), _stream())
    return h, gu, hw


def grouped_gemm_down(h, offsets, down, H):
    """y_perm [R, H] bf16."""
    _need(h, "h", _BF16, 2)
    _need(down, "down", _BF16, 2)
    R, I = h.shape
    E = down.shape[0] // I
    if down.shape != (E * I, H):
        raise ValueError("down must be [E*I, H]")
    if offsets is not None:
        _need(offsets, "offsets", torch.int32, 1)
    y = torch.empty((R, H), dtype=_BF16, device=h.device)
    call("moe_grouped_gemm_down", _p(h), _p(offsets), _p(down), R, H, E, I, _p(y), _stream())
    return y


def unpermute_combine(y_perm, row_map, w, y_shared=None, out=None):
    """y [T, H] bf16 (out: an existing contiguous [T, H] bf16 tensor or row slice to write)."""
    _need(y_perm, "y_perm", _BF16, 2)
    _need(row_map, "row_map", torch.int32, 1)
    _need(w, "w", torch.float32, 2)
    if y_shared is not None:
        _need(y_shared, "y_shared", _BF16, 2)
    T, k = w.shape
    H = y_perm.shape[1]
    if out is None:
        y = torch.empty((T, H), dtype=_BF16, device=y_perm.device)
    else:
        _need(out, "out", _BF16, 2)
        if tuple(out.shape) != (T, H):
            raise ValueError("out must be [T, H]")
        y = out
    call("moe_unpermute_combine", _p(y_perm), _p(row_map), _p(w), _p(y_shared), T, H, k, _p(y), _stream())
    return y


# ---------------------------------------------------------------- backward

def unpermute_combine_bwd(dy, src_row):
    """dy_perm [R, H] bf16: the dY row of each permuted row (unweighted, exact)."""
    _need(dy, "dy", _BF16, 2)
    _need(src_row, "src_row", torch.int32, 1)
    T, H = dy.shape
    R = src_row.shape[0]
    if (T == 0) != (R == 0) or (T > 0 and R % T):
        raise ValueError("src_row must hold T*k rows for dy [T, H]")
    k = R // T if T > 0 else 1   # an empty batch: any k >= 1 describes it
    dy_perm = torch.empty((R, H), dtype=_BF16, device=dy.device)
    call("moe_unpermute_combine_bwd", _p(dy), _p(src_row), T, H, k, _p(dy_perm), _stream())
    return dy_perm


def down_bwd_parts(I):
    n = ctypes.c_int64(0)
    call("moe_grouped_gemm_down_bwd_parts", I, ctypes.byref(n))
    return n.value


def grouped_gemm_down_bwd(dy_perm, h_w, gu_pre, w_perm, offsets, down):
    """dgu [R, 2I] bf16, d_down [E*I, H] bf16, dw_part [R, nparts] fp32."""
    _need(dy_perm, "dy_perm", _BF16, 2)
    _need(h_w, "h_w", _BF16, 2)
    _need(gu_pre, "gu_pre", torch.float32, 2)
    _need(w_perm, "w_perm", torch.float32, 1)
    _need(down, "down", _BF16, 2)
    R, I = h_w.shape
    H = dy_perm.shape[1]
    E = down.shape[0] // I
    if offsets is not None:
        _need(offsets, "offsets", torch.int32, 1)
    dgu = torch.empty((R, 2 * I), dtype=_BF16, device=h_w.device)
    d_down = torch.empty((E * I, H), dtype=_BF16, device=h_w.device)
    parts = torch.empty((R, down_bwd_parts(I)), dtype=torch.float32, device=h_w.device)
    call("moe_grouped_gemm_down_bwd", _p(dy_perm), _p(h_w), _p(gu_pre), _p(w_perm), _p(offsets), _p(down), R,
         H, E, I, _p(dgu), _p(d_down), _p(parts), _stream())
    return dgu, d_down, parts


def route_bwd(dw_part, row_map, w, ids, E):
    """d_logits [T, E] fp32 and dw [T, k] fp32 from the per-row partials of the down backward."""
    _need(dw_part, "dw_part", torch.float32, 2)
    _need(row_map, "row_map", torch.int32, 1)
    _need(w, "w", torch.float32, 2)
    _need(ids, "ids", torch.int32, 2)
    T, k = w.shape
    dl = torch.empty((T, E), dtype=torch.float32, device=w.device)
    dw = torch.empty((T, k), dtype=torch.float32, device=w.device)
    call("moe_route_bwd", _p(dw_part), dw_part.shape[1], _p(row_map), _p(w), _p(ids), T, E, k, _p(dl), _p(dw),
         _stream())
    return dl, dw


def grouped_gemm_gate_up_bwd(dgu, x, src_row, offsets, gate_up):
    """dx_perm [R, H] bf16, d_gate_up [E*H, 2I] bf16."""
    _need(dgu, "dgu", _BF16, 2)
    _need(x, "x", _BF16, 2)
    _need(gate_up, "gate_up", _BF16, 2)
    R, I2 = dgu.shape
    I = I2 // 2
    T, H = x.shape
    E = gate_up.shape[0] // H
    if src_row is not None:
        _need(src_row, "src_row", torch.int32, 1)
    if offsets is not None:
        _need(offsets, "offsets", torch.int32, 1)
    dx_perm = torch.empty((R, H), dtype=_BF16, device=x.device)
    d_gu = torch.empty((E * H, 2 * I), dtype=_BF16, device=x.device)
    call("moe_grouped_gemm_gate_up_bwd", _p(dgu), _p(x), _p(src_row), _p(offsets), _p(gate_up), T, R, H, E,
         I, _p(dx_perm), _p(d_gu), _stream())
    return dx_perm, d_gu


def gather_dx(dx_perm, row_map, T, k, d_logits=None, ids=None, w_router=None):
    """dX [T, H] bf16 = sum_j dx_perm[row_map] (+ d_logits . W_r^T on the chosen experts)."""
    _need(dx_perm, "dx_perm", _BF16, 2)
    _need(row_map, "row_map", torch.int32, 1)
    H = dx_perm.shape[1]
    E = 1
    ws = None
    if d_logits is not None:
        _need(d_logits, "d_logits", torch.float32, 2)
        _need(ids, "ids", torch.int32, 2)
        _need(w_router, "w_router", torch.float32, 2)
        E = w_router.shape[1]
        nbytes = ctypes.c_size_t(0)
        call("moe_gather_dx_workspace_size", H, E, ctypes.byref(nbytes))
        ws = _ws(nbytes.value, dx_perm.device)
    else:
        E = max(k, 1)
    dx = torch.empty((T, H), dtype=_BF16, device=dx_perm.device)
    call("moe_gather_dx", _p(dx_perm), _p(row_map), _p(d_logits), _p(ids), _p(w_router), T, H, E, k, _p(dx),
         _p(ws), 0 if ws is None else ws.numel(), _stream())
    return dx


def route_bwd_weight(x, d_logits):
    """d_w_router [H, E] fp32 = x^T . d_logits."""
    _need(x, "x", _BF16, 2)
    _need(d_logits, "d_logits", torch.float32, 2)
    T, H = x.shape
    E = d_logits.shape[1]
    out = torch.empty((H, E), dtype=torch.float32, device=x.device)
    call("moe_route_bwd_weight", _p(x), _p(d_logits), T, H, E, _p(out), _stream())
    return out
