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


def test_gemm_wait_runs_out_and_context_survives():
    moe = lib()
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
    h, _, _ = moe.grouped_gemm_gate_up_swiglu(bf(x), None, None, bf(gu), I)
    y = moe.grouped_gemm_down(h, None, bf(dn), H)
    moe.sync_status()
    assert_close("dense FFN after the timeout", f64(y), oracle.dense_ffn(x, gu, dn))
