"""GPU parity of the expert-parallel pieces (through the C ABI): the chunk
transpose of the dispatch and combine, the replica map of EPLB-style
replication, and the layer with experts split over G ranks emulated on one
GPU ("Awesome-ML-SYS-Tutorial" MoE/EP guide, gsyq.cn, "Expert Parallelism";
hotspot experts and EPLB).  Integer outputs are compared bit for bit with
the oracle; the emulated expert-parallel layer must equal the local layer
bit for bit (every expert sees the same rows in the same order) and the
oracle within the parity tolerance."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import bf, f32, f64, i32, lib, npi
from parity import TIE_TAU, assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("A,B,zero_frac,seed", [(1, 1, 0.0, 0), (2, 8, 0.2, 1), (8, 16, 0.5, 2),
                                                (8, 8, 0.0, 3), (64, 256, 0.3, 4), (16, 1, 0.0, 5),
                                                (3, 1000, 0.9, 6)])
def test_sort_chunks_matches_oracle(A, B, zero_frac, seed):
    """src_of, pos_of and the group offsets bit for bit against the oracle's
    chunk transpose: empty chunks, a single chunk, 64 x 256 chunks (the
    receiver's (source, local expert) matrix of 64 ranks and 256 experts)."""
    moe = lib()
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, 40, size=(A, B)).astype(np.int32)
    counts[rng.random((A, B)) < zero_frac] = 0
    N = int(counts.sum())
    src_of, pos_of, group = moe.ops.sort_chunks(i32(counts), N)
    moe.sync_status()
    ref = oracle.sort_chunks(counts)
    np.testing.assert_array_equal(npi(src_of), ref[0], err_msg="src_of")
    np.testing.assert_array_equal(npi(pos_of), ref[1], err_msg="pos_of")
    np.testing.assert_array_equal(npi(group), ref[2], err_msg="group offsets")


def test_sort_chunks_reports_counts_that_do_not_sum_to_n():
    """Counts that do not sum to N are reported (MOE_ERR_DEVICE) and nothing
    is written past the N rows."""
    import torch
    moe = lib()
    counts = i32(np.array([[3, 4], [5, 6]], dtype=np.int32))
    for N in (10, 20):   # the counts sum to 18
        guard = torch.full((N + 8,), -5, dtype=torch.int32, device=counts.device)
        group = torch.empty(3, dtype=torch.int32, device=counts.device)
        nbytes = __import__("ctypes").c_size_t(0)
        moe.ops.call("moe_sort_chunks_workspace_size", 2, 2, __import__("ctypes").byref(nbytes))
        ws = torch.empty(max(nbytes.value, 16), dtype=torch.uint8, device=counts.device)
        pos = torch.empty(N, dtype=torch.int32, device=counts.device)
        moe.ops.call("moe_sort_chunks", moe.ops._p(counts), 2, 2, N, moe.ops._p(guard), moe.ops._p(pos),
                     moe.ops._p(group), moe.ops._p(ws), ws.numel(), moe.ops._stream())
        with pytest.raises(moe.MoEError) as ei:
            moe.sync_status()
        assert ei.value.status == 6
        assert (npi(guard)[N:] == -5).all()


def test_map_replicas_matches_oracle():
    moe = lib()
    rng = np.random.default_rng(7)
    T, k, E, G = 1000, 4, 16, 4
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    load = np.bincount(ids.reshape(-1), minlength=E)
    plan = oracle.eplb_plan(load, G, E + 8)
    got = moe.ops.ep_map_replicas(i32(ids), i32(plan["rep_first"]), i32(plan["rep_count"]), i32(plan["rep_list"]))
    moe.sync_status()
    np.testing.assert_array_equal(npi(got), oracle.map_replicas(ids, plan["rep_first"], plan["rep_count"],
                                                                 plan["rep_list"]))


def _layer_inputs(moe, cfg):
    inp = synth.make_inputs(cfg)
    return inp, bf(inp.x), f32(inp.w_router), bf(inp.gate_up), bf(inp.down), \
        (f32(inp.bias) if inp.bias is not None else None)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_ep_emulated_equals_local_layer(G):
    """The layer with experts split over G ranks (every rank's steps run on
    this GPU, the all-to-alls as chunk transposes) equals moe_forward bit for
    bit, and the oracle within the tolerance; T = 300 tokens do not split
    evenly over the ranks."""
    import torch
    from token_dispatch_grouped_softmax_gb300 import ep
    moe = lib()
    cfg = synth.MoEConfig("ep", T=300, H=256, E=16, k=4, I=128, seed=40 + G)
    inp, x, wr, gu, dn, _ = _layer_inputs(moe, cfg)
    stats = {}
    y_ep = ep.ep_forward_emulated(x, wr, gu, dn, cfg.k, G, stats=stats)
    y_local, _ = moe.moe_forward(x, wr, gu, dn, cfg.k)
    moe.sync_status()
    assert torch.equal(y_ep.view(torch.int16), y_local.view(torch.int16))
    assert stats["rows_per_rank"].sum() == cfg.R
    r = oracle.route(inp.x, inp.w_router, None, cfg.k)
    zk = np.abs(r["logits"][np.arange(cfg.T), r["ids"][:, -1]])
    assert np.all(np.minimum(r["kgap"], r["ordgap"]) > TIE_TAU * np.maximum(1.0, zk))
    assert_close("y (EP emulated, G=%d)" % G, f64(y_ep), oracle.layer_forward(inp)["y"])


def test_ep_emulated_qwen3_moe_shape():
    """The Qwen3-MoE-shaped workload (T = 4096, E = 128) over 8 ranks: equal
    to the local layer bit for bit."""
    import torch
    from token_dispatch_grouped_softmax_gb300 import ep
    moe = lib()
    cfg = synth.CONFIGS["qwen3_moe"]
    inp, x, wr, gu, dn, _ = _layer_inputs(moe, cfg)
    y_ep = ep.ep_forward_emulated(x, wr, gu, dn, cfg.k, 8)
    y_local, _ = moe.moe_forward(x, wr, gu, dn, cfg.k)
    moe.sync_status()
    assert torch.equal(y_ep.view(torch.int16), y_local.view(torch.int16))


def test_eplb_replicas_balance_skewed_routing():
    """The skewed workload (hotspot experts, empty experts) over 8 ranks:
    with an EPLB-style plan from the expert loads (32 extra replicas) the
    output is still the local layer's bit for bit, and the busiest rank's
    rows drop from 1.41x the mean (the plain split of experts) to within 10%
    of it."""
    import torch
    from token_dispatch_grouped_softmax_gb300 import ep
    moe = lib()
    cfg = synth.CONFIGS["qwen3_moe_skewed"]
    inp, x, wr, gu, dn, bias = _layer_inputs(moe, cfg)
    y_local, st = moe.moe_forward(x, wr, gu, dn, cfg.k, bias)
    load = npi(st.counts).astype(np.int64)
    G = 8
    plain = {}
    y_plain = ep.ep_forward_emulated(x, wr, gu, dn, cfg.k, G, bias=bias, stats=plain)
    plan = ep.EPLBPlan.build(load, G, cfg.E + 32)
    weights = ep.replicate_weights(gu, dn, plan.phys_to_log)
    balanced = {}
    y_bal = ep.ep_forward_emulated(x, wr, gu, dn, cfg.k, G, bias=bias, plan=plan, phys_weights=weights,
                                   stats=balanced)
    moe.sync_status()
    for y in (y_plain, y_bal):
        assert torch.equal(y.view(torch.int16), y_local.view(torch.int16))
    mean = cfg.R / G
    print("busiest rank / mean: plain %.2f, EPLB %.2f" % (plain["rows_per_rank"].max() / mean,
                                                        balanced["rows_per_rank"].max() / mean))
    assert plain["rows_per_rank"].max() > 1.3 * mean        # the hotspots overload one rank (1.41x)
    assert balanced["rows_per_rank"].max() < 1.1 * mean     # the plan spreads them (1.0x planned)


@pytest.mark.parametrize("G", [1, 2, 8])
def test_ep_fused_dispatch_equals_local_layer(G):
    """The receivers' gate_up GEMMs gather their rows straight from the
    senders' token rows (no dispatch copy, no re-sort copy): the local
    layer's output bit for bit, at T = 300 tokens (uneven token ranges) and
    at the Qwen3-MoE shape over 8 ranks."""
    import torch
    from token_dispatch_grouped_softmax_gb300 import ep
    moe = lib()
    for cfg in (synth.MoEConfig("ep", T=300, H=256, E=16, k=4, I=128, seed=60 + G), synth.CONFIGS["qwen3_moe"]):
        if cfg.E % G:
            continue
        inp, x, wr, gu, dn, _ = _layer_inputs(moe, cfg)
        y_fused = ep.ep_forward_emulated(x, wr, gu, dn, cfg.k, G, fused_dispatch=True)
        y_local, _ = moe.moe_forward(x, wr, gu, dn, cfg.k)
        moe.sync_status()
        assert torch.equal(y_fused.view(torch.int16), y_local.view(torch.int16)), cfg.name


def test_ep_fused_dispatch_with_eplb_replicas():
    """The fused dispatch over physical experts (EPLB replicas of the skewed
    workload's hotspots), equal to the local layer bit for bit."""
    import torch
    from token_dispatch_grouped_softmax_gb300 import ep
    moe = lib()
    cfg = synth.CONFIGS["qwen3_moe_skewed"]
    inp, x, wr, gu, dn, bias = _layer_inputs(moe, cfg)
    y_local, st = moe.moe_forward(x, wr, gu, dn, cfg.k, bias)
    plan = ep.EPLBPlan.build(npi(st.counts).astype(np.int64), 8, cfg.E + 32)
    weights = ep.replicate_weights(gu, dn, plan.phys_to_log)
    y = ep.ep_forward_emulated(x, wr, gu, dn, cfg.k, 8, bias=bias, plan=plan, phys_weights=weights,
                               fused_dispatch=True)
    moe.sync_status()
    assert torch.equal(y.view(torch.int16), y_local.view(torch.int16))
