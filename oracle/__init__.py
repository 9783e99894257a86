"""fp64 CPU oracle of the MoE expert layer (ctypes wrapper of moe_oracle.c).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this package.  It shares no code with the
CUDA path and imports nothing from it.

Every function takes numpy arrays.  Inputs come either as the synthetic
workloads' raw encodings (bf16 bits as uint16 for x / gate_up / down / dY /
shared weights, fp32 for W_r and bias), which are widened exactly, or all as
float64 (used by the finite-difference pins).  All arithmetic is fp64.

Every function is pinned by tests/test_oracle_pins.py (the expert-parallel
index functions by tests/test_oracle_ep_pins.py); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "moe_oracle.c"), os.path.join(_HERE, "moe_oracle_body.h")]
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into liboracle.so (in place) when missing or stale."""
    newest = max(os.path.getmtime(s) for s in _SRCS)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", _SRCS[0], "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_P = ctypes.c_void_p
_I = ctypes.c_int64

_SIGS = {
    "oracle_route": [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "oracle_dense_ffn": [_I, _I, _I, _P, _P, _P, _P],
    "oracle_forward_permuted": [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P,
                                _P, _P, _P, _P, _P],
    "oracle_forward_dense": [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, _P],
    "oracle_forward_tokens": [_I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P],
    "oracle_backward_tokens": [_I, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "oracle_backward_expert": [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P],
    "oracle_backward": [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
}


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        for base, sig in _SIGS.items():
            for suf in ("_bits", "_f64"):
                f = getattr(lib, base + suf)
                f.argtypes = sig
                f.restype = None
        lib.oracle_permute.argtypes = [_I, _I, _I, _P, _P, _P, _P, _P]
        lib.oracle_permute.restype = ctypes.c_int
        lib.oracle_permute_rows.argtypes = [_I, _I, _P, _P, _P]
        lib.oracle_permute_rows.restype = None
        lib.oracle_unpermute_combine.argtypes = [_I, _I, _I, _P, _P, _P, _P, _P]
        lib.oracle_unpermute_combine.restype = None
        lib.oracle_threads.argtypes = []
        lib.oracle_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def threads():
    """OpenMP threads the oracle's parallel loops run on."""
    return int(_load().oracle_threads())


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _variant(*acts):
    """'_bits' when the activation/weight arrays are bf16 bits, '_f64' for doubles."""
    kinds = {a.dtype for a in acts if a is not None}
    if kinds == {np.dtype(np.uint16)}:
        return "_bits"
    if kinds == {np.dtype(np.float64)}:
        return "_f64"
    raise TypeError("oracle inputs must be all bf16 bits (uint16) or all float64, got %s" % kinds)


def _router_arr(a, suffix):
    if a is None:
        return None
    want = np.float32 if suffix == "_bits" else np.float64
    assert a.dtype == want, "router arrays must be %s for this variant" % np.dtype(want)
    return np.ascontiguousarray(a)


def _f(name, suffix):
    return getattr(_load(), name + suffix)


# --------------------------------------------------------------------- router

def route(x, w_r, bias, k):
    """Router: fp64 logits, softmax, top-k (ties to the lower index), renormalised weights.

    Returns dict(ids [T,k] int32, w [T,k] f64, logits [T,E], probs [T,E], kgap [T], ordgap [T]).
    """
    T, H = x.shape
    E = w_r.shape[1]
    sfx = _variant(x)
    w_r = _router_arr(w_r, sfx)
    bias = _router_arr(bias, sfx)
    out = dict(ids=np.empty((T, k), np.int32), w=np.empty((T, k)), logits=np.empty((T, E)),
               probs=np.empty((T, E)), kgap=np.empty(T), ordgap=np.empty(T))
    _f("oracle_route", sfx)(T, H, E, k, _ptr(x), _ptr(w_r), _ptr(bias), _ptr(out["logits"]),
                            _ptr(out["probs"]), _ptr(out["ids"]), _ptr(out["w"]), _ptr(out["kgap"]),
                            _ptr(out["ordgap"]))
    return out


def weights_for_ids(logits, ids):
    """Renormalised gate weights of a given expert choice, from fp64 logits.

    The router's last step ("InternVL3.5 接入 pure FSDP2 后端开发实践" §8.2:
    gate -> FP32 softmax -> top-k -> 权重归一化): w_j = p_{e_j} / sum_i p_{e_i}
    with p = softmax(logits).  The softmax denominator cancels, so this is the
    softmax over the chosen logits alone; it is evaluated that way (shifted by
    their maximum).  Used where the experts chosen for a token are given (for
    instance by the device's fp32 router at an fp32-vs-fp64 near tie), so
    that everything downstream of the choice can be checked for that choice.

    logits [T, E] float64, ids [T, k] int -> w [T, k] float64.
    """
    logits = np.asarray(logits, dtype=np.float64)
    ids = np.asarray(ids, dtype=np.int64)
    z = np.take_along_axis(logits, ids, axis=1)
    e = np.exp(z - z.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


# -------------------------------------------------------------------- permute

def permute(ids, E):
    """Per-expert counts, exclusive-scan offsets, stable row_map and src_row."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    R = T * k
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    row_map = np.empty(R, np.int32)
    src_row = np.empty(R, np.int32)
    rc = _load().oracle_permute(T, k, E, _ptr(ids), _ptr(counts), _ptr(offsets), _ptr(row_map),
                                _ptr(src_row))
    if rc != 0:
        raise ValueError("expert id out of range")
    return dict(counts=counts, offsets=offsets, row_map=row_map, src_row=src_row)


def permute_rows(x, src_row):
    """x_perm[row] = x[src_row[row]] (float64)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    src_row = np.ascontiguousarray(src_row, dtype=np.int32)
    R, H = src_row.shape[0], x.shape[1]
    out = np.empty((R, H))
    _load().oracle_permute_rows(R, H, _ptr(x), _ptr(src_row), _ptr(out))
    return out


def unpermute_combine(y_perm, row_map, w, y_shared=None):
    """y[t] = sum_j w[t,j] * y_perm[row_map[t*k+j]] (+ y_shared[t]) (float64)."""
    y_perm = np.ascontiguousarray(y_perm, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    row_map = np.ascontiguousarray(row_map, dtype=np.int32)
    T, k = w.shape
    H = y_perm.shape[1]
    if y_shared is not None:
        y_shared = np.ascontiguousarray(y_shared, dtype=np.float64)
    y = np.empty((T, H))
    _load().oracle_unpermute_combine(T, k, H, _ptr(y_perm), _ptr(row_map), _ptr(w), _ptr(y_shared),
                                     _ptr(y))
    return y


# -------------------------------------------------------------------- forward

def dense_ffn(x, gu, dn):
    """A dense SwiGLU FFN on every row of x: gu [H, 2I], dn [I, H]."""
    T, H = x.shape
    I = dn.shape[0]
    sfx = _variant(x, gu, dn)
    y = np.empty((T, H))
    _f("oracle_dense_ffn", sfx)(T, H, I, _ptr(x), _ptr(gu), _ptr(dn), _ptr(y))
    return y


def forward_permuted(x, gate_up, down, w, perm, k, sh_gu=None, sh_dn=None, want_intermediates=False):
    """The permuted-form forward.  perm is the dict from ``permute``."""
    T, H = x.shape
    E = perm["counts"].shape[0]
    I = down.shape[0] // E
    R = T * k
    I_s = sh_dn.shape[0] if sh_dn is not None else 0
    sfx = _variant(x, gate_up, down, sh_gu, sh_dn)
    w = np.ascontiguousarray(w, dtype=np.float64)
    y = np.empty((T, H))
    extra = {}
    if want_intermediates:
        extra = dict(gu_perm=np.empty((R, 2 * I)), h_perm=np.empty((R, I)), y_perm=np.empty((R, H)))
        if I_s:
            extra["y_shared"] = np.empty((T, H))
    _f("oracle_forward_permuted", sfx)(
        T, H, E, k, I, _ptr(x), _ptr(gate_up), _ptr(down), _ptr(w), _ptr(perm["offsets"]),
        _ptr(perm["row_map"]), _ptr(perm["src_row"]), I_s, _ptr(sh_gu), _ptr(sh_dn),
        _ptr(extra.get("gu_perm")), _ptr(extra.get("h_perm")), _ptr(extra.get("y_perm")),
        _ptr(extra.get("y_shared")), _ptr(y))
    if want_intermediates:
        return y, extra
    return y


def forward_dense(x, gate_up, down, ids, w, sh_gu=None, sh_dn=None):
    """Brute force: every expert on every token, masked by the routing."""
    T, H = x.shape
    k = ids.shape[1]
    E = gate_up.shape[0] // H
    I = down.shape[0] // E
    I_s = sh_dn.shape[0] if sh_dn is not None else 0
    sfx = _variant(x, gate_up, down, sh_gu, sh_dn)
    y = np.empty((T, H))
    _f("oracle_forward_dense", sfx)(T, H, E, k, I, _ptr(x), _ptr(gate_up), _ptr(down),
                                    _ptr(np.ascontiguousarray(ids, np.int32)),
                                    _ptr(np.ascontiguousarray(w, np.float64)), I_s, _ptr(sh_gu),
                                    _ptr(sh_dn), _ptr(y))
    return y


def forward_tokens(tokens, x, gate_up, down, ids, w, sh_gu=None, sh_dn=None, want_f=False):
    """The per-token definition on a token list; returns y [n, H] (and f [n, k, H])."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    n = tokens.shape[0]
    T, H = x.shape
    k = ids.shape[1]
    E = gate_up.shape[0] // H
    I = down.shape[0] // E
    I_s = sh_dn.shape[0] if sh_dn is not None else 0
    sfx = _variant(x, gate_up, down, sh_gu, sh_dn)
    y = np.empty((n, H))
    f = np.empty((n, k, H)) if want_f else None
    _f("oracle_forward_tokens", sfx)(n, _ptr(tokens), H, E, k, I, _ptr(x), _ptr(gate_up), _ptr(down),
                                     _ptr(np.ascontiguousarray(ids, np.int32)),
                                     _ptr(np.ascontiguousarray(w, np.float64)), I_s, _ptr(sh_gu),
                                     _ptr(sh_dn), _ptr(y), _ptr(f))
    return (y, f) if want_f else y


# ------------------------------------------------------------------- backward

def backward(x, w_r, gate_up, down, ids, w, dy, want_dw=True, want_dwr=False):
    """Full analytic backward of L = sum <dY, y>: dict(dX, dlogits, dw, d_gate_up, d_down, d_w_r)."""
    T, H = x.shape
    k = ids.shape[1]
    E = w_r.shape[1]
    I = down.shape[0] // E
    sfx = _variant(x, gate_up, down, dy)
    w_r = _router_arr(w_r, sfx)
    out = dict(dX=np.empty((T, H)), dlogits=np.empty((T, E)), dw=np.empty((T, k)))
    if want_dw:
        out["d_gate_up"] = np.empty((E * H, 2 * I))
        out["d_down"] = np.empty((E * I, H))
    if want_dwr:
        out["d_w_r"] = np.empty((H, E))
    _f("oracle_backward", sfx)(T, H, E, k, I, _ptr(x), _ptr(w_r), _ptr(gate_up), _ptr(down),
                               _ptr(np.ascontiguousarray(ids, np.int32)),
                               _ptr(np.ascontiguousarray(w, np.float64)), _ptr(dy), _ptr(out["dX"]),
                               _ptr(out["dlogits"]), _ptr(out["dw"]), _ptr(out.get("d_gate_up")),
                               _ptr(out.get("d_down")), _ptr(out.get("d_w_r")))
    return out


def backward_tokens(tokens, x, w_r, gate_up, down, ids, w, dy):
    """dX [n, H], dlogits [n, E], dw [n, k] for a token list."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int64)
    n = tokens.shape[0]
    T, H = x.shape
    k = ids.shape[1]
    E = w_r.shape[1]
    I = down.shape[0] // E
    sfx = _variant(x, gate_up, down, dy)
    w_r = _router_arr(w_r, sfx)
    dX, dl, dw = np.empty((n, H)), np.empty((n, E)), np.empty((n, k))
    _f("oracle_backward_tokens", sfx)(n, _ptr(tokens), H, E, k, I, _ptr(x), _ptr(w_r),
                                      _ptr(gate_up), _ptr(down),
                                      _ptr(np.ascontiguousarray(ids, np.int32)),
                                      _ptr(np.ascontiguousarray(w, np.float64)), _ptr(dy), _ptr(dX),
                                      _ptr(dl), _ptr(dw))
    return dict(dX=dX, dlogits=dl, dw=dw)


def backward_expert(e, x, gate_up, down, ids, w, dy):
    """d_gate_up_e [H, 2I] and d_down_e [I, H] of one expert."""
    T, H = x.shape
    k = ids.shape[1]
    E = gate_up.shape[0] // H
    I = down.shape[0] // E
    sfx = _variant(x, gate_up, down, dy)
    dgu = np.empty((H, 2 * I))
    ddn = np.empty((I, H))
    _f("oracle_backward_expert", sfx)(int(e), T, H, k, I, _ptr(x), _ptr(gate_up), _ptr(down),
                                      _ptr(np.ascontiguousarray(ids, np.int32)),
                                      _ptr(np.ascontiguousarray(w, np.float64)), _ptr(dy), _ptr(dgu),
                                      _ptr(ddn))
    return dgu, ddn


# --------------------------------------------------------------- whole layer

def layer_forward(inp, want_intermediates=False):
    """Route -> permute -> experts -> combine on a synth.MoEInputs (full size)."""
    cfg = inp.cfg
    r = route(inp.x, inp.w_router, inp.bias, cfg.k)
    perm = permute(r["ids"], cfg.E)
    res = forward_permuted(inp.x, inp.gate_up, inp.down, r["w"], perm, cfg.k, inp.sh_gate_up,
                           inp.sh_down, want_intermediates=want_intermediates)
    if want_intermediates:
        y, extra = res
    else:
        y, extra = res, {}
    return dict(route=r, perm=perm, y=y, **extra)


# ------------------------------------------------------- expert parallelism
# The index flow of expert-parallel dispatch and combine (Awesome-ML-SYS-
# Tutorial MoE/EP guide, gsyq.cn, "Expert Parallelism": dispatch by
# all-to-all with split sizes from the per-expert token counts, the
# receiver's re-sort of its chunks by local expert, combine by all-to-all;
# hotspot experts and EPLB-style replication), as plain loops.

def sort_chunks(counts):
    """Rows in an A x B matrix of chunks, row-major (a, b) order, reordered to
    (b, a) order, each chunk's rows kept in order.  Returns src_of [N] (the
    input row at each output position), pos_of [N] (its inverse) and
    group_offsets [B+1] (the first output row of each b)."""
    counts = np.asarray(counts, dtype=np.int64)
    A, B = counts.shape
    start = {}
    n = 0
    for a in range(A):
        for b in range(B):
            start[(a, b)] = n
            n += int(counts[a, b])
    src_of, group = [], []
    for b in range(B):
        group.append(len(src_of))
        for a in range(A):
            for l in range(int(counts[a, b])):
                src_of.append(start[(a, b)] + l)
    group.append(len(src_of))
    src_of = np.array(src_of, dtype=np.int32)
    pos_of = np.empty_like(src_of)
    pos_of[src_of] = np.arange(len(src_of), dtype=np.int32)
    return src_of, pos_of, np.array(group, dtype=np.int32)


def map_replicas(ids, rep_first, rep_count, rep_list):
    """Assignment (t, j) of logical expert e goes to its replica t mod
    rep_count[e]: physical expert rep_list[rep_first[e] + t % rep_count[e]]."""
    ids = np.asarray(ids)
    out = np.empty_like(ids, dtype=np.int32)
    T, k = ids.shape
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            out[t, j] = rep_list[rep_first[e] + t % rep_count[e]]
    return out


def eplb_plan(load, G, n_phys):
    """EPLB-style replication and placement, the greedy steps in order: extra
    replicas one at a time to the expert with the largest load per replica
    (lower index on ties); replica loads by the round-robin split (load //
    rep, the first load % rep replicas one more); replicas heaviest first
    (then lower expert, lower replica) to the least-loaded rank with a free
    slot (n_phys // G each; lower rank on ties); physical ids rank-major,
    within a rank by (expert, replica)."""
    from fractions import Fraction
    load = [int(v) for v in load]
    E = len(load)
    rep = [1] * E
    for _ in range(n_phys - E):
        best = max(range(E), key=lambda e: (Fraction(load[e], rep[e]), -e))
        rep[best] += 1
    reps = [(load[e] // rep[e] + (1 if r < load[e] % rep[e] else 0), e, r) for e in range(E) for r in range(rep[e])]
    reps.sort(key=lambda x: (-x[0], x[1], x[2]))
    slots = n_phys // G
    rank_load, used, on = [0] * G, [0] * G, [[] for _ in range(G)]
    for ld, e, r in reps:
        g = min((c for c in range(G) if used[c] < slots), key=lambda c: (rank_load[c], c))
        rank_load[g] += ld
        used[g] += 1
        on[g].append((e, r))
    rep_first = np.cumsum([0] + rep[:-1]).astype(np.int32)
    rep_list = np.empty(n_phys, np.int32)
    phys_to_log = np.empty(n_phys, np.int32)
    for g in range(G):
        for i, (e, r) in enumerate(sorted(on[g])):
            p = g * slots + i
            phys_to_log[p] = e
            rep_list[rep_first[e] + r] = p
    return dict(phys_to_log=phys_to_log, rep_first=rep_first, rep_count=np.array(rep, np.int32),
                rep_list=rep_list, rank_load=np.array(rank_load, np.int64))


def ep_dispatch(ids_per_rank, n_phys, G):
    """The rows each EP rank's experts receive.  ids_per_rank[s]: the (physical)
    expert ids [T_s, k] of source rank s; rank d owns experts [d P, (d+1) P),
    P = n_phys // G.  Returns, per destination d, a list of (source, token,
    slot) in the order its local experts see them (local expert, then source,
    then the source's stable permuted order) and its local expert offsets
    [P+1]."""
    P = n_phys // G
    out = []
    for d in range(G):
        rows, offs = [], []
        for p in range(P):
            e = d * P + p
            offs.append(len(rows))
            for s, ids in enumerate(ids_per_rank):
                perm = permute(ids, n_phys)
                assignment = np.empty_like(perm["row_map"])     # permuted row -> assignment i = t k + j
                assignment[perm["row_map"]] = np.arange(perm["row_map"].shape[0], dtype=np.int32)
                for row in range(perm["offsets"][e], perm["offsets"][e + 1]):
                    i = int(assignment[row])
                    rows.append((s, i // ids.shape[1], i % ids.shape[1]))
        offs.append(len(rows))
        out.append((rows, np.array(offs, dtype=np.int32)))
    return out
