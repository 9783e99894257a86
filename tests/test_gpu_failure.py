"""Failure detection on the GPU without a fault: a bounded wait that runs out.

With the test hook on, the grouped GEMM's producer issues no loads, so the
MMA warp's wait on its first stage can never complete.  The wait is bounded
(here 50 ms): the kernel records MOE_ERR_TIMEOUT in the status word, stops its
other warps, frees its tensor memory and returns; the host reads the status,
and the same context then runs a normal call correctly.  Nothing traps,
faults or spins unbounded.
"""
import pytest

import oracle
import synth
from gpu_helpers import bf, f64, lib
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pairs", [0, 2], ids=["single", "pairs"])
def test_gemm_wait_runs_out_and_context_survives(pairs):
    """On single CTAs and on CTA pairs (both CTAs of a pair run their own
    bounded waits and meet at the final cluster barrier)."""
    moe = lib()
    moe.set_gemm_pairs(pairs)
    L = moe.load()
    T, H, I = 256, 128, 64
    x = synth.normal_bf16(31, synth.TID_X, (T, H), 1.0)
    gu = synth.normal_bf16(31, synth.TID_SH_GATE_UP, (H, 2 * I), H ** -0.5)
    moe.sync_status()
    moe.set_wait_limit_ns(50_000_000)
    L.moe_test_stall_gemm_producer(1)
    try:
        moe.grouped_gemm_gate_up_swiglu(bf(x), None, None, bf(gu), I)
        with pytest.raises(moe.MoEError) as ei:
            moe.sync_status()
        assert ei.value.status == 4   # MOE_ERR_TIMEOUT
    finally:
        L.moe_test_stall_gemm_producer(0)
        moe.set_wait_limit_ns(0)
    moe.sync_status()                 # the status word was cleared
    dn = synth.normal_bf16(31, synth.TID_SH_DOWN, (I, H), I ** -0.5)
    try:
        h, _, _ = moe.grouped_gemm_gate_up_swiglu(bf(x), None, None, bf(gu), I)
        y = moe.grouped_gemm_down(h, None, bf(dn), H)
        moe.sync_status()
    finally:
        moe.set_gemm_pairs(moe.GEMM_PAIRS_GATE_UP)
    assert_close("dense FFN after the timeout", f64(y), oracle.dense_ffn(x, gu, dn))


def _expect_device_error(moe):
    with pytest.raises(moe.MoEError) as ei:
        moe.sync_status()
    assert ei.value.status == 6   # MOE_ERR_DEVICE
    moe.sync_status()             # the status word was cleared


def test_bad_indices_are_reported_not_followed():
    """Index data that no permutation produces (a combine / gather_dx row
    outside the permuted rows, a dY source row outside the tokens, an expert
    id outside [0, E), expert offsets that are not a scan of counts ending at
    R) is reported as MOE_ERR_DEVICE; the kernels read a valid row instead or
    do no work, so nothing faults and the context stays usable."""
    import torch
    moe = lib()
    dev = torch.device("cuda", 0)
    T, H, E, k, I = 64, 128, 8, 2, 64
    R = T * k
    yp = torch.zeros((R, H), dtype=torch.bfloat16, device=dev)
    w = torch.full((T, k), 0.5, dtype=torch.float32, device=dev)
    good = torch.arange(R, dtype=torch.int32, device=dev)
    moe.sync_status()
    for bad_row in (R, -1):
        rm = good.clone()
        rm[17] = bad_row
        moe.unpermute_combine(yp, rm, w)
        _expect_device_error(moe)
        moe.gather_dx(yp, rm, T, k)
        _expect_device_error(moe)
    src = (good // k).clone()
    src[5] = T                          # one past the last token
    moe.unpermute_combine_bwd(torch.zeros((T, H), dtype=torch.bfloat16, device=dev), src)
    _expect_device_error(moe)
    wr = torch.zeros((H, E), dtype=torch.float32, device=dev)
    ids = torch.zeros((T, k), dtype=torch.int32, device=dev)
    ids[3, 1] = E
    dl = torch.zeros((T, E), dtype=torch.float32, device=dev)
    moe.gather_dx(yp, good, T, k, dl, ids, wr)
    _expect_device_error(moe)
    x = torch.zeros((R, H), dtype=torch.bfloat16, device=dev)
    gu = torch.zeros((E * H, 2 * I), dtype=torch.bfloat16, device=dev)
    for offs in ([0, 40, 30, 60, 80, 100, 110, 120, R], [0, 16, 32, 48, 64, 80, 96, 112, R + 16],
                 [4, 16, 32, 48, 64, 80, 96, 112, R]):
        offsets = torch.tensor(offs, dtype=torch.int32, device=dev)
        moe.grouped_gemm_gate_up_swiglu(x, None, offsets, gu, I)
        _expect_device_error(moe)
    # the context still computes correctly
    ok_offsets = torch.arange(0, R + 1, R // E, dtype=torch.int32, device=dev)
    h, _, _ = moe.grouped_gemm_gate_up_swiglu(x, None, ok_offsets, gu, I)
    moe.sync_status()
    assert bool((h.float() == 0).all())
