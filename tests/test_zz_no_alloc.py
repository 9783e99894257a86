"""moe_permute_noalloc against moe_permute, through the C ABI.

moe_permute_noalloc is for callers that cannot allocate device memory at the
moment they route tokens: a plugin running inside an inference engine's
enqueue step (which must not allocate), a runtime that has reserved all
device memory for its own pool, or a latency-critical path that cannot pay
for cudaMalloc's implicit synchronisation.  Its scratch is a fixed array
inside the library instead of a caller workspace.  This file checks that two
calls in a row give exactly what moe_permute gives with its own workspace
and what the fp64 oracle's permutation gives, and that sizes beyond the
fixed scratch are refused.  It is kept in a file of
its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import dev, f32, i32, lib, npi

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p
MOE_ERR_SCRATCH_LIMIT = 7


def _p(t):
    return None if t is None else P(t.data_ptr())


def _outputs(T, k, E, with_w):
    d = dev()
    R = T * k
    return dict(counts=torch.empty(E, dtype=torch.int32, device=d),
                offsets=torch.empty(E + 1, dtype=torch.int32, device=d),
                row_map=torch.empty(R, dtype=torch.int32, device=d),
                src_row=torch.empty(R, dtype=torch.int32, device=d),
                w_perm=torch.empty(R, dtype=torch.float32, device=d) if with_w else None)


def _stream():
    return P(torch.cuda.current_stream().cuda_stream)


def _permute_with_workspace(L, ids, w, E):
    T, k = ids.shape
    o = _outputs(T, k, E, w is not None)
    n = ctypes.c_size_t(0)
    assert L.moe_permute_workspace_size(T, k, E, ctypes.byref(n)) == 0
    ws = torch.empty(max(n.value, 16), dtype=torch.uint8, device=dev())
    rc = L.moe_permute(_p(ids), _p(w), T, k, E, _p(o["counts"]), _p(o["offsets"]), _p(o["row_map"]),
                       _p(o["src_row"]), _p(o["w_perm"]), _p(ws), ws.numel(), _stream())
    assert rc == 0
    return o


def _permute_noalloc(L, ids, w, E):
    T, k = ids.shape
    o = _outputs(T, k, E, w is not None)
    rc = L.moe_permute_noalloc(_p(ids), _p(w), T, k, E, _p(o["counts"]), _p(o["offsets"]),
                               _p(o["row_map"]), _p(o["src_row"]), _p(o["w_perm"]), _stream())
    assert rc == 0
    return o


def test_noalloc_matches_permute_on_two_calls_in_a_row():
    moe = lib()
    L = moe.load()
    cases = []
    for T, k, E, seed in ((4096, 8, 128, 1), (777, 6, 1000, 2)):
        ids_h = synth.distinct_ids(seed, synth.TID_IDS, T, k, E)
        w_h = np.random.default_rng(seed).uniform(0.0, 1.0, (T, k)).astype(np.float32)
        ids, w = i32(ids_h), f32(w_h)
        cases.append((ids_h, w_h, ids, w, E, _permute_with_workspace(L, ids, w, E)))
    got = [_permute_noalloc(L, ids, w, E) for _, _, ids, w, E, _ in cases]   # two calls in a row
    moe.sync_status()
    for (ids_h, w_h, ids, w, E, ref), out in zip(cases, got):
        perm = oracle.permute(ids_h, E)
        for key in ("counts", "offsets", "row_map", "src_row"):
            np.testing.assert_array_equal(npi(out[key]), perm[key], err_msg=key + " vs the oracle")
        w_perm = np.empty(ids_h.size, dtype=np.float32)
        w_perm[perm["row_map"]] = w_h.reshape(-1)   # each assignment's weight at its permuted row
        np.testing.assert_array_equal(npi(out["w_perm"]), w_perm, err_msg="w_perm vs the oracle")
        for key in ("counts", "offsets", "row_map", "src_row", "w_perm"):
            np.testing.assert_array_equal(npi(out[key]), npi(ref[key]), err_msg=key)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    L = lib().load()
    fake = P(0x10000)   # never dereferenced: the call is refused before anything is enqueued
    T, k, E = 2048 * 1025 // 8, 8, 1024   # ceil(T*k / 2048) * E = 1025 * 1024 > 2^20
    rc = L.moe_permute_noalloc(fake, None, T, k, E, fake, fake, fake, fake, None, None)
    assert rc == MOE_ERR_SCRATCH_LIMIT
    assert L.moe_error_string(rc) == b"size exceeds the fixed scratch of moe_permute_noalloc"
