"""GPU parity of the grouped GEMMs and the whole layer, forward and backward,
against the fp64 oracle (through the C ABI).

Small cases are compared element by element; they span several 128- and
256-row tiles (the latter once experts average 512 rows), 256-column tiles,
ragged expert tails of one and two 128-row halves, empty experts, and partial
column tiles.  The named workloads (Qwen3-MoE shape, skewed routing, the training
step, DeepSeek-V3 shape) run at full size in the launch configuration the
benchmark times and are compared on seeded token / expert samples the oracle
computes one by one; their integer outputs are compared in full.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import bf, f32, f64, i32, lib, npi
from parity import TIE_TAU, U_BF16, assert_close, bf16_allowance, compare_ids, sample_tokens

pytestmark = pytest.mark.gpu

SMALL = [
    # T, H, E, k, I
    (64, 128, 8, 2, 64),        # the tiny workload's shapes
    (200, 128, 8, 2, 128),      # ragged expert tails
    (512, 256, 16, 4, 192),     # I = 192: a partial gate/up column tile
    (300, 384, 6, 3, 320),      # H = 384: a partial 256-column output tile
    (50, 128, 64, 1, 64),       # mostly empty experts
    (1100, 256, 4, 2, 128),     # >= 512 rows per expert: 256-row tiles, one-half tails
    (1400, 384, 4, 2, 192),     # 256-row tiles with two-half tails, partial column tiles
]


def _inputs(T, H, E, k, I, seed, **kw):
    cfg = synth.MoEConfig("c", T=T, H=H, E=E, k=k, I=I, seed=seed, **kw)
    return cfg, synth.make_inputs(cfg, with_dy=True)


def _forward(moe, inp, save=False, fused="rows"):
    """fused: "tma" gathers the token rows inside the gate_up GEMM (TMA
    tile::gather4); "rows" materialises them first."""
    x, wr = bf(inp.x), f32(inp.w_router)
    gu, dn = bf(inp.gate_up), bf(inp.down)
    bias = f32(inp.bias) if inp.bias is not None else None
    sgu = bf(inp.sh_gate_up) if inp.sh_gate_up is not None else None
    sdn = bf(inp.sh_down) if inp.sh_down is not None else None
    y, st = moe.moe_forward(x, wr, gu, dn, inp.cfg.k, bias, sgu, sdn, save_for_backward=save,
                            fused_gather=fused != "rows")
    moe.sync_status()
    return (x, wr, gu, dn), y, st


@pytest.mark.parametrize("fused", ["tma", "rows"])
@pytest.mark.parametrize("T,H,E,k,I", SMALL)
def test_forward_elementwise(T, H, E, k, I, fused):
    moe = lib()
    cfg, inp = _inputs(T, H, E, k, I, seed=T + H + I)
    _, y, st = _forward(moe, inp, save=True, fused=fused)
    ref = oracle.layer_forward(inp, want_intermediates=True)
    same, tol = compare_ids(npi(st.ids), ref["route"])
    assert tol == 0 and same.all()
    for key in ("counts", "offsets", "row_map", "src_row"):
        np.testing.assert_array_equal(npi(getattr(st, key)), ref["perm"][key], err_msg=key)
    w_perm_ref = np.empty(cfg.R)
    w_perm_ref[ref["perm"]["row_map"]] = ref["route"]["w"].reshape(-1)
    assert_close("w_perm", f64(st.w_perm), w_perm_ref, bf16_out=False)
    assert_close("gu_pre", f64(st.gu_pre), ref["gu_perm"], bf16_out=False)
    assert_close("h", f64(st.h), ref["h_perm"])
    assert_close("h_w", f64(st.h_w), w_perm_ref[:, None] * ref["h_perm"])
    assert_close("y_perm", f64(st.y_perm), ref["y_perm"])
    assert_close("y", f64(y), ref["y"])


@pytest.mark.parametrize("T,H,I", [(256, 128, 64), (300, 256, 192), (129, 512, 1024)])
def test_dense_mode_is_one_swiglu_ffn(T, H, I):
    """src_row = offsets = NULL, E = 1: the shared-expert (dense) mode."""
    moe = lib()
    x = synth.normal_bf16(T, synth.TID_X, (T, H), 1.0)
    gu = synth.normal_bf16(T, synth.TID_SH_GATE_UP, (H, 2 * I), H ** -0.5)
    dn = synth.normal_bf16(T, synth.TID_SH_DOWN, (I, H), I ** -0.5)
    h, _, _ = moe.grouped_gemm_gate_up_swiglu(bf(x), None, None, bf(gu), I)
    y = moe.grouped_gemm_down(h, None, bf(dn), H)
    moe.sync_status()
    assert_close("dense ffn", f64(y), oracle.dense_ffn(x, gu, dn))


def test_shared_expert_layer():
    moe = lib()
    cfg, inp = _inputs(300, 256, 8, 2, 128, seed=21, I_shared=256)
    _, y, st = _forward(moe, inp)
    ref = oracle.layer_forward(inp)
    same, tol = compare_ids(npi(st.ids), ref["route"])
    assert tol == 0
    assert_close("y", f64(y), ref["y"])


@pytest.mark.parametrize("fused", ["tma", "rows"])
@pytest.mark.parametrize("T,H,E,k,I", SMALL)
def test_backward_elementwise(T, H, E, k, I, fused):
    moe = lib()
    cfg, inp = _inputs(T, H, E, k, I, seed=3 * T + I)
    (x, wr, gu, dn), y, st = _forward(moe, inp, save=True, fused=fused)
    g = moe.moe_backward(bf(inp.dy), st, wr, gu, dn, want_dw_router=True)
    moe.sync_status()
    r = oracle.route(inp.x, inp.w_router, None, k)
    same, tol = compare_ids(npi(st.ids), r)
    assert tol == 0 and same.all()
    b = oracle.backward(inp.x, inp.w_router, inp.gate_up, inp.down, r["ids"], r["w"], inp.dy,
                        want_dw=True, want_dwr=True)
    assert_close("dw", f64(g["dw"]), b["dw"], bf16_out=False)
    assert_close("d_logits", f64(g["d_logits"]), b["dlogits"], bf16_out=False)
    assert_close("dX", f64(g["dx"]), b["dX"])
    assert_close("d_gate_up", f64(g["d_gate_up"]), b["d_gate_up"])
    assert_close("d_down", f64(g["d_down"]), b["d_down"])
    assert_close("d_w_router", f64(g["d_w_router"]), b["d_w_r"], bf16_out=False)


@pytest.mark.parametrize("T,H,E,k,I", [(200, 320, 256, 8, 64), (1000, 192, 128, 8, 64), (64, 128, 256, 12, 64),
                                     (40, 128, 512, 6, 64)])
def test_backward_dx_router_term_shapes(T, H, E, k, I):
    """dX with the router term (d_logits . W_r^T on the chosen experts) and
    d_logits against the oracle's backward at expert counts the layer tests
    do not reach: E = 256 (k = 8 and k = 12), E = 128 with 1000 tokens, and
    E = 512 (the split-K router)."""
    moe = lib()
    cfg, inp = _inputs(T, H, E, k, I, seed=11 * T + E)
    (x, wr, gu, dn), y, st = _forward(moe, inp, save=True)
    g = moe.moe_backward(bf(inp.dy), st, wr, gu, dn)
    moe.sync_status()
    r = oracle.route(inp.x, inp.w_router, None, k)
    same, tol = compare_ids(npi(st.ids), r)
    assert same.all(), "near-tie routing at a small shape"
    b = oracle.backward(inp.x, inp.w_router, inp.gate_up, inp.down, r["ids"], r["w"], inp.dy, want_dw=False)
    assert_close("d_logits", f64(g["d_logits"]), b["dlogits"], bf16_out=False)
    assert_close("dX", f64(g["dx"]), b["dX"])


def test_dy_rows_gather_equals_scatter():
    """The combine's backward moves dY rows to permuted order: the gather
    (moe_unpermute_combine_bwd, by src_row) and the token-by-token scatter
    the layer uses (moe_permute_rows_scatter, by row_map) give the same bits,
    and the oracle's rows."""
    import torch
    moe = lib()
    cfg, inp = _inputs(300, 256, 16, 4, 64, seed=17)
    (x, wr, gu, dn), y, st = _forward(moe, inp, save=True)
    dy = bf(inp.dy)
    a = moe.ops.unpermute_combine_bwd(dy, st.src_row)
    b = moe.ops.permute_rows_scatter(dy, st.row_map, cfg.k)
    moe.sync_status()
    assert torch_equal(a, b)
    np.testing.assert_array_equal(f64(b), oracle.permute_rows(synth.bf16_to_f32(inp.dy), npi(st.src_row)))


def test_backward_empty_experts_get_zero_weight_grads():
    moe = lib()
    cfg, inp = _inputs(40, 128, 32, 1, 64, seed=5)
    (x, wr, gu, dn), y, st = _forward(moe, inp, save=True)
    g = moe.moe_backward(bf(inp.dy), st, wr, gu, dn)
    moe.sync_status()
    counts = npi(st.counts)
    empty = np.nonzero(counts == 0)[0]
    assert empty.size > 0
    dgu = f64(g["d_gate_up"]).reshape(32, 128, 128)
    ddn = f64(g["d_down"]).reshape(32, 64, 128)
    assert not dgu[empty].any() and not ddn[empty].any()


def test_every_token_on_the_same_two_experts():
    """Degenerate routing: a router bias of +40 on experts 2 and 7 sends every
    token to those two (in either order), so six experts are empty and two
    hold T rows each; forward and backward element by element against the
    oracle, and zero weight gradients for the empty experts."""
    moe = lib()
    T, H, E, k, I = 300, 128, 8, 2, 64
    cfg, inp = _inputs(T, H, E, k, I, seed=17)
    inp.bias = np.zeros(E, dtype=np.float32)
    inp.bias[[2, 7]] = 40.0
    (x, wr, gu, dn), y, st = _forward(moe, inp, save=True)
    g = moe.moe_backward(bf(inp.dy), st, wr, gu, dn, want_dw_router=True)
    moe.sync_status()
    assert npi(st.counts).tolist() == [0, 0, T, 0, 0, 0, 0, T]
    assert (np.sort(npi(st.ids), axis=1) == np.array([2, 7])).all()
    ref = oracle.layer_forward(inp, want_intermediates=True)
    same, tol = compare_ids(npi(st.ids), ref["route"])
    assert tol == 0 and same.all()
    np.testing.assert_array_equal(npi(st.row_map), ref["perm"]["row_map"])
    assert_close("y", f64(y), ref["y"])
    r = ref["route"]
    b = oracle.backward(inp.x, inp.w_router, inp.gate_up, inp.down, r["ids"], r["w"], inp.dy,
                        want_dw=True, want_dwr=True)
    assert_close("dw", f64(g["dw"]), b["dw"], bf16_out=False)
    assert_close("d_logits", f64(g["d_logits"]), b["dlogits"], bf16_out=False)
    assert_close("dX", f64(g["dx"]), b["dX"])
    assert_close("d_w_router", f64(g["d_w_router"]), b["d_w_r"], bf16_out=False)
    # weight gradients per expert block, as in the sampled training test
    # (six of the eight blocks are exact zeros and would halve a whole-tensor RMS)
    dgu = f64(g["d_gate_up"]).reshape(E, H, 2 * I)
    ddn = f64(g["d_down"]).reshape(E, I, H)
    rgu = b["d_gate_up"].reshape(E, H, 2 * I)
    rdn = b["d_down"].reshape(E, I, H)
    for e in (2, 7):
        assert_close("d_gate_up[%d]" % e, dgu[e], rgu[e])
        assert_close("d_down[%d]" % e, ddn[e], rdn[e])
    empty = [0, 1, 3, 4, 5, 6]
    assert not dgu[empty].any() and not ddn[empty].any()


def test_empty_batch_forward_backward():
    """T = 0: every call is a no-op that still writes what it owes: zero
    counts and offsets, zero weight gradients, [0, H] outputs."""
    import torch
    moe = lib()
    H, E, k, I = 128, 8, 2, 64
    cfg, inp = _inputs(64, H, E, k, I, seed=11)
    wr, gu, dn = f32(inp.w_router), bf(inp.gate_up), bf(inp.down)
    x = torch.empty((0, H), dtype=torch.bfloat16, device=wr.device)
    y, st = moe.moe_forward(x, wr, gu, dn, k, save_for_backward=True)
    moe.sync_status()
    assert tuple(y.shape) == (0, H)
    assert not npi(st.counts).any() and not npi(st.offsets).any()
    g = moe.moe_backward(torch.empty((0, H), dtype=torch.bfloat16, device=wr.device), st, wr, gu, dn,
                         want_dw_router=True)
    moe.sync_status()
    assert tuple(g["dx"].shape) == (0, H) and tuple(g["d_logits"].shape) == (0, E)
    for name in ("d_gate_up", "d_down", "d_w_router"):
        assert not f64(g[name]).any(), name


def _permutation_of_gpu_ids(st, E):
    """The permutation is a pure integer function of the routing ids:
    counts, offsets, row_map and src_row must equal, bit for bit, the
    oracle's permutation of the ids the GPU chose, whatever near ties the
    GPU's fp32 router took either way."""
    gids = npi(st.ids)
    perm = oracle.permute(gids, E)
    for key in ("counts", "offsets", "row_map", "src_row"):
        np.testing.assert_array_equal(npi(getattr(st, key)), perm[key], err_msg=key)
    return gids, perm


def _sampled_forward_check(cfg_name, n_tokens=None, fused="rows", max_tied=None):
    """The named workload at full size: routing ids against the oracle's (near
    ties counted), the permutation bit-exact against the oracle's permutation
    of the GPU's ids, the gate weights against the oracle's weights for the
    GPU's choice, and y on n_tokens seeded tokens (None: every token) against
    the oracle computed for that choice."""
    moe = lib()
    cfg = synth.CONFIGS[cfg_name]
    inp = synth.make_inputs(cfg)
    _, y, st = _forward(moe, inp, fused=fused)
    r = oracle.route(inp.x, inp.w_router, inp.bias, cfg.k)
    same, tol = compare_ids(npi(st.ids), r, label=cfg_name)
    assert tol <= (max(4, cfg.T // 2000) if max_tied is None else max_tied)
    gids, _ = _permutation_of_gpu_ids(st, cfg.E)
    w_ref = oracle.weights_for_ids(r["logits"], gids)
    assert_close("w (%s)" % cfg_name, f64(st.w), w_ref, bf16_out=False)
    tok = np.arange(cfg.T) if n_tokens is None else sample_tokens(cfg.T, n_tokens, cfg.seed)
    yref = oracle.forward_tokens(tok, inp.x, inp.gate_up, inp.down, gids, w_ref, inp.sh_gate_up,
                                 inp.sh_down)
    assert_close("y (%s)" % cfg_name, f64(y)[tok], yref)
    return st


@pytest.mark.parametrize("fused", ["rows", "tma"])
def test_qwen3_moe_forward_full(fused):
    """Every token of the Qwen3-MoE-shaped workload."""
    _sampled_forward_check("qwen3_moe", fused=fused)


def test_skewed_routing_forward_full():
    """Every token of the skewed workload (hotspot and empty experts)."""
    st = _sampled_forward_check("qwen3_moe_skewed")
    counts = npi(st.counts)
    assert (counts == 0).sum() >= 8


def test_deepseek_v3_forward_sampled():
    """1,024 seeded tokens of the DeepSeek-V3-shaped workload (with its
    shared expert); the permutation in full."""
    _sampled_forward_check("deepseek_v3", n_tokens=1024)


def test_training_step_backward_sampled():
    """The training workload (T = 8192) forward with saved activations and
    backward.  dX, d_logits and dw on 1,024 seeded tokens, and the weight
    gradients of 8 whole experts (the busiest, the least busy and 6 seeded
    others), all against the oracle evaluated for the experts the GPU chose,
    so every check runs whatever near ties the fp32 router took."""
    moe = lib()
    cfg = synth.CONFIGS["qwen3_moe_train"]
    inp = synth.make_inputs(cfg)
    (x, wr, gu, dn), y, st = _forward(moe, inp, save=True)
    g = moe.moe_backward(bf(inp.dy), st, wr, gu, dn)
    moe.sync_status()
    r = oracle.route(inp.x, inp.w_router, None, cfg.k)
    same, tol = compare_ids(npi(st.ids), r, label="qwen3_moe_train")
    assert tol <= max(4, cfg.T // 2000)
    gids, perm = _permutation_of_gpu_ids(st, cfg.E)
    w_ref = oracle.weights_for_ids(r["logits"], gids)
    tok = sample_tokens(cfg.T, 1024, 33)
    yref = oracle.forward_tokens(tok, inp.x, inp.gate_up, inp.down, gids, w_ref)
    assert_close("y (train)", f64(y)[tok], yref)
    b = oracle.backward_tokens(tok, inp.x, inp.w_router, inp.gate_up, inp.down, gids, w_ref, inp.dy)
    assert_close("dX (train)", f64(g["dx"])[tok], b["dX"])
    assert_close("d_logits (train)", f64(g["d_logits"])[tok], b["dlogits"], bf16_out=False)
    assert_close("dw (train)", f64(g["dw"])[tok], b["dw"], bf16_out=False)
    H, I = cfg.H, cfg.I
    counts = perm["counts"]
    rng = np.random.default_rng(cfg.seed)
    busiest, idlest = int(np.argmax(counts)), int(np.argmin(counts))
    others = [e for e in rng.permutation(cfg.E).tolist() if e not in (busiest, idlest)][:6]
    experts = [busiest, idlest] + others
    assert len(set(experts)) == 8
    dgu, ddn = g["d_gate_up"], g["d_down"]
    for e in experts:
        rgu, rdn = oracle.backward_expert(e, inp.x, inp.gate_up, inp.down, gids, w_ref, inp.dy)
        assert_close("d_gate_up[e] (train)", f64(dgu[e * H:(e + 1) * H]), rgu)
        assert_close("d_down[e] (train)", f64(ddn[e * I:(e + 1) * I]), rdn)


def _oracle_y(inp, x_bits):
    """The oracle's layer output for the tokens x_bits with inp's weights;
    asserts first that no token sits within the near-tie band of the routing
    comparison (TIE_TAU, relative), where the fp32 device router must choose
    as the fp64 oracle does."""
    k = inp.cfg.k
    r = oracle.route(x_bits, inp.w_router, inp.bias, k)
    zk = np.abs(r["logits"][np.arange(x_bits.shape[0]), r["ids"][:, -1]])
    assert np.all(np.minimum(r["kgap"], r["ordgap"]) > TIE_TAU * np.maximum(1.0, zk))
    perm = oracle.permute(r["ids"], inp.cfg.E)
    return oracle.forward_permuted(x_bits, inp.gate_up, inp.down, r["w"], perm, k, inp.sh_gate_up,
                                   inp.sh_down)


def torch_equal(a, b):
    import torch
    return bool(torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                            b.view(torch.uint8) if b.dtype == torch.bfloat16 else b))


def test_forward_graph_router_split_refresh():
    """A ForwardGraph makes W_r's bf16 split once; after W_r changes in place,
    refresh_router_split() makes the replays follow the new router (against
    the oracle and bit for bit against moe_forward)."""
    import torch
    moe = lib()
    cfg, inp = _inputs(300, 256, 16, 2, 128, seed=95)
    wr, gu, dn = f32(inp.w_router), bf(inp.gate_up), bf(inp.down)
    g = moe.ForwardGraph(300, wr, gu, dn, cfg.k)
    xb = synth.normal_bf16(8, synth.TID_X, (300, 256), 1.0)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    new_wr = synth.normal_f32(96, synth.TID_WR, (256, 16), 256 ** -0.5)
    wr.copy_(torch.from_numpy(new_wr).cuda())
    g.refresh_router_split()
    y_graph = g(x).clone()
    y_eager, _ = moe.moe_forward(x, wr, gu, dn, cfg.k)
    moe.sync_status()
    assert torch_equal(y_graph, y_eager)
    inp2 = synth.MoEInputs(inp.cfg, inp.x, new_wr, None, inp.gate_up, inp.down)
    assert_close("y (ForwardGraph, new W_r)", f64(y_graph), _oracle_y(inp2, xb))


def test_pipelined_forward_matches_forward():
    """PipelinedForward (copies overlapped with the layer on two streams):
    every batch's output against the oracle, and bit for bit equal to
    moe_forward's."""
    import torch
    moe = lib()
    cfg, inp = _inputs(256, 256, 8, 2, 128, seed=77)
    wr, gu, dn = f32(inp.w_router), bf(inp.gate_up), bf(inp.down)
    xbits = [synth.normal_bf16(s, synth.TID_X, (256, 256), 1.0) for s in (1, 2, 3)]
    xs = [torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory() for xb in xbits]
    ys = [torch.empty((256, 256), dtype=torch.bfloat16).pin_memory() for _ in xs]
    moe.PipelinedForward(256, wr, gu, dn, cfg.k).run(xs, ys)
    moe.sync_status()
    for xb, xh, yh in zip(xbits, xs, ys):
        assert_close("y (PipelinedForward)", f64(yh), _oracle_y(inp, xb))
        y, _ = moe.moe_forward(xh.cuda(), wr, gu, dn, cfg.k)
        assert torch_equal(y.cpu(), yh)


def test_forward_graph_replays_match_forward():
    """ForwardGraph: one capture, replayed on new tokens (new routing each
    time): each replay's output against the oracle, and bit for bit equal to
    moe_forward's, the shared expert included."""
    import torch
    moe = lib()
    cfg, inp = _inputs(300, 256, 8, 2, 128, seed=91, I_shared=64)
    wr, gu, dn = f32(inp.w_router), bf(inp.gate_up), bf(inp.down)
    sgu, sdn = bf(inp.sh_gate_up), bf(inp.sh_down)
    g = moe.ForwardGraph(300, wr, gu, dn, cfg.k, None, sgu, sdn)
    for s in (5, 6, 7):
        xb = synth.normal_bf16(s, synth.TID_X, (300, 256), 1.0)
        x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        y_graph = g(x).clone()
        moe.sync_status()
        assert_close("y (ForwardGraph)", f64(y_graph), _oracle_y(inp, xb))
        y_eager, _ = moe.moe_forward(x, wr, gu, dn, cfg.k, None, sgu, sdn)
        moe.sync_status()
        assert torch_equal(y_graph, y_eager)


@pytest.mark.parametrize("fused", ["rows", "tma"])
@pytest.mark.parametrize("T,H,E,k,I", SMALL + [(4096, 256, 16, 2, 192)])
def test_cta_pairs_bit_identical(T, H, E, k, I, fused):
    """The grouped GEMMs on CTA pairs (2-SM MMAs, 256-row tiles, M = 128 pair
    MMAs for tails of up to 128 rows; the weight-gradient GEMMs with their K
    tails zeroed by each CTA of the pair) give the single-CTA results bit for
    bit: forward with saved activations and the whole backward."""
    import torch
    moe = lib()
    cfg, inp = _inputs(T, H, E, k, I, seed=5 * T + I)
    outs = []
    for pairs in (moe.GEMM_PAIRS_NONE, moe.GEMM_PAIRS_ALL, moe.GEMM_PAIRS_GATE_UP_WGRAD):
        moe.set_gemm_pairs(pairs)
        try:
            (x, wr, gu, dn), y, st = _forward(moe, inp, save=True, fused=fused)
            g = moe.moe_backward(bf(inp.dy), st, wr, gu, dn)
            moe.sync_status()
        finally:
            moe.set_gemm_pairs(moe.GEMM_PAIRS_GATE_UP)
        outs.append([y, st.h, st.gu_pre, st.h_w, st.y_perm] + [g[n] for n in sorted(g)])
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch_equal(a, b)


@pytest.mark.parametrize("T,H,E,k,I", [(300, 384, 6, 3, 320), (1100, 256, 4, 2, 128)])
def test_programmatic_launch_bit_identical(T, H, E, k, I):
    """Kernels launched with and without programmatic dependent launch (each
    kernel's set-up overlapping the previous kernel's tail) give the same
    forward and backward bit for bit."""
    moe = lib()
    cfg, inp = _inputs(T, H, E, k, I, seed=7 * T + I)
    outs = []
    for pdl in (True, False):
        moe.set_pdl(pdl)
        try:
            (x, wr, gu, dn), y, st = _forward(moe, inp, save=True)
            g = moe.moe_backward(bf(inp.dy), st, wr, gu, dn, want_dw_router=True)
            moe.sync_status()
        finally:
            moe.set_pdl(True)
        outs.append([y, st.ids, st.row_map, st.h, st.gu_pre, st.y_perm] + [g[n] for n in sorted(g)])
    for a, b in zip(*outs):
        assert torch_equal(a, b)


def test_overlapped_forward_matches_forward():
    """OverlappedForward (route/permute of batch i+1 overlapping the expert
    GEMMs of batch i, on two streams): every batch's output against the
    oracle, and bit for bit equal to moe_forward's, with and without a shared
    expert and with the row gather fused into the gate_up GEMM (both read x
    inside the expert stage)."""
    import torch
    moe = lib()
    for I_s, fused in ((0, False), (64, False), (0, True)):
        cfg, inp = _inputs(300, 256, 8, 2, 128, seed=93, I_shared=I_s)
        wr, gu, dn = f32(inp.w_router), bf(inp.gate_up), bf(inp.down)
        sgu = bf(inp.sh_gate_up) if I_s else None
        sdn = bf(inp.sh_down) if I_s else None
        xbits = [synth.normal_bf16(s, synth.TID_X, (300, 256), 1.0) for s in (11, 12, 13, 14, 15)]
        xs = [torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory() for xb in xbits]
        ys = [torch.empty((300, 256), dtype=torch.bfloat16).pin_memory() for _ in xs]
        moe.OverlappedForward(300, wr, gu, dn, cfg.k, None, sgu, sdn, fused_gather=fused).run(xs, ys)
        moe.sync_status()
        for xb, yh in zip(xbits, ys):
            assert_close("y (OverlappedForward)", f64(yh), _oracle_y(inp, xb))
        for xh, yh in zip(xs, ys):
            y, _ = moe.moe_forward(xh.cuda(), wr, gu, dn, cfg.k, None, sgu, sdn)
            assert torch_equal(y.cpu(), yh)



# expert sizes around every tile boundary of the grouped GEMMs: empty
# experts, 1 row, 16-row steps, 64-row boxes, 128-row tiles and their tails,
# 256-row tiles (two halves) and their tails
TILE_EDGE_COUNTS = [0, 1, 15, 16, 17, 63, 64, 65, 80, 127, 128, 129, 200, 255, 256, 257, 300, 383, 384,
                    385, 511, 512, 513, 700, 1000, 0, 33]
# at least 512 rows per expert on average: the down GEMM's 256-row tiles with
# one- and two-half tails
HEAVY_COUNTS = [513, 1000, 0, 700, 1024, 2047]


@pytest.mark.parametrize("pairs", [False, True], ids=["single", "pairs"])
@pytest.mark.parametrize("counts", [TILE_EDGE_COUNTS, HEAVY_COUNTS], ids=["edges", "heavy"])
@pytest.mark.parametrize("H,I", [(256, 192), (320, 128)])
def test_grouped_gemms_at_tile_edges(H, I, counts, pairs):
    """The forward grouped GEMMs on explicit expert offsets whose sizes sit on
    either side of every tile boundary (I = 192: a partial gate/up column
    tile; H = 320: a partial down output tile), element by element against
    the oracle (identity permutation, k = 1); on single CTAs and on CTA pairs
    (256-row tiles, tails of up to 128 rows as M = 128 pair MMAs)."""
    moe = lib()
    E, R = len(counts), sum(counts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = synth.normal_bf16(R + H, synth.TID_X, (R, H), 1.0)
    gu = synth.normal_bf16(R + H, synth.TID_GATE_UP, (E * H, 2 * I), H ** -0.5)
    dn = synth.normal_bf16(R + H, synth.TID_DOWN, (E * I, H), I ** -0.5)
    ident = np.arange(R, dtype=np.int32)
    perm = dict(counts=np.array(counts, dtype=np.int32), offsets=offs, row_map=ident,
                src_row=ident)
    _, ref = oracle.forward_permuted(x, gu, dn, np.ones((R, 1)), perm, 1, want_intermediates=True)
    moe.set_gemm_pairs(pairs)
    try:
        h, _, _ = moe.grouped_gemm_gate_up_swiglu(bf(x), None, i32(offs), bf(gu), I)
        y = moe.grouped_gemm_down(h, i32(offs), bf(dn), H)
        moe.sync_status()
    finally:
        moe.set_gemm_pairs(moe.GEMM_PAIRS_GATE_UP)
    assert_close("h", f64(h), ref["h_perm"])
    assert_close("y_perm", f64(y), ref["y_perm"])


@pytest.mark.parametrize("counts", [TILE_EDGE_COUNTS, HEAVY_COUNTS], ids=["edges", "heavy"])
@pytest.mark.parametrize("H,I", [(256, 192), (320, 128)])
def test_weight_gradients_at_tile_edges(H, I, counts):
    """The weight-gradient GEMMs, whose K is an expert's rows, on expert sizes
    either side of every 64-row K block (and empty experts): on single CTAs
    (two 128-row halves) and on CTA pairs (each CTA zeroes its own stage's
    rows past the expert), bit for bit the same; and against the expert
    blocks of the oracle's backward (identity permutation, k = 1).  H = 320
    and I = 192 leave the last 256-row tile with 64 rows, which the second
    CTA of a pair has none of."""
    import torch
    moe = lib()
    E, R = len(counts), sum(counts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = synth.normal_bf16(R + I, synth.TID_X, (R, H), 1.0)
    gu = synth.normal_bf16(R + I, synth.TID_GATE_UP, (E * H, 2 * I), H ** -0.5)
    dn = synth.normal_bf16(R + I, synth.TID_DOWN, (E * I, H), I ** -0.5)
    dy = synth.normal_bf16(R + I, synth.TID_DY, (R, H), 1.0)
    ids = np.repeat(np.arange(E, dtype=np.int32), counts).reshape(R, 1)
    w1 = np.ones((R, 1))
    ref = oracle.backward(x, np.zeros((H, E), np.float32), gu, dn, ids, w1, dy)
    xb, dyb = bf(x), bf(dy)
    outs = []
    for pairs in (moe.GEMM_PAIRS_GATE_UP, moe.GEMM_PAIRS_GATE_UP_WGRAD):
        moe.set_gemm_pairs(pairs)
        try:
            w_perm = torch.ones(R, dtype=torch.float32, device=xb.device)
            h, gu_pre, h_w = moe.grouped_gemm_gate_up_swiglu(xb, None, i32(offs), bf(gu), I, w_perm=w_perm,
                                                             save_for_backward=True)
            dgu, d_down, _ = moe.grouped_gemm_down_bwd(dyb, h_w, gu_pre, w_perm, i32(offs), bf(dn))
            _, d_gu = moe.grouped_gemm_gate_up_bwd(dgu, xb, None, i32(offs), bf(gu))
            moe.sync_status()
        finally:
            moe.set_gemm_pairs(moe.GEMM_PAIRS_GATE_UP)
        outs.append((d_down, d_gu))
    for a, b in zip(*outs):
        assert torch_equal(a, b)
    assert_close("d_down", f64(outs[1][0]), ref["d_down"])
    assert_close("d_gate_up", f64(outs[1][1]), ref["d_gate_up"])


def _sweep_shapes(n, seed):
    """n seeded layer shapes off the hand-picked ones: odd and prime expert
    counts (2 to 256, so the fused router, the split-K router and the
    cluster permute's chunk sizes all turn up), k from 1 to 8, T from 1 to
    700 (ragged 128-row tiles and expert tails), H and I from 64 to 448."""
    rng = np.random.default_rng(seed)
    shapes = []
    for _ in range(n):
        E = int(rng.choice([2, 3, 5, 7, 12, 16, 24, 31, 48, 64, 100, 128, 160, 256]))
        k = int(rng.integers(1, min(E, 8) + 1))
        shapes.append((int(rng.integers(1, 701)), 64 * int(rng.integers(1, 8)), E, k, 64 * int(rng.integers(1, 8))))
    return shapes


@pytest.mark.parametrize("T,H,E,k,I", _sweep_shapes(16, 20261202))
def test_seeded_shape_sweep_forward_backward(T, H, E, k, I):
    """Forward (saving activations) and backward through the layer at seeded
    irregular shapes, every output against the oracle: the ids bit for bit
    up to the stated near-tie rule, the permutation bit for bit against the
    oracle's permutation of the GPU's ids, y and all gradients element by
    element for the experts the GPU chose."""
    moe = lib()
    cfg, inp = _inputs(T, H, E, k, I, seed=T * 7 + E * 13 + k)
    (x, wr, gu, dn), y, st = _forward(moe, inp, save=True)
    g = moe.moe_backward(bf(inp.dy), st, wr, gu, dn, want_dw_router=True)
    moe.sync_status()
    r = oracle.route(inp.x, inp.w_router, None, k)
    same, tol = compare_ids(npi(st.ids), r, label="sweep")
    assert tol <= 1
    gids, perm = _permutation_of_gpu_ids(st, E)
    w_ref = oracle.weights_for_ids(r["logits"], gids)
    assert_close("w", f64(st.w), w_ref, bf16_out=False)
    ref = oracle.forward_permuted(inp.x, inp.gate_up, inp.down, w_ref, perm, k)
    assert_close("y", f64(y), ref)
    b = oracle.backward(inp.x, inp.w_router, inp.gate_up, inp.down, gids, w_ref, inp.dy, want_dw=True,
                        want_dwr=True)
    assert_close("dX", f64(g["dx"]), b["dX"])
    assert_close("d_logits", f64(g["d_logits"]), b["dlogits"], bf16_out=False)
    assert_close("dw", f64(g["dw"]), b["dw"], bf16_out=False)
    assert_close("d_w_router", f64(g["d_w_router"]), b["d_w_r"], bf16_out=False)
    # The weight gradients are sums over an expert's rows (here as few as 1 to
    # 14) of products with one rounded bf16 operand, dgu or w h: their
    # allowance uses u * sum|a||b| over those products (see parity.py), from
    # the operands as the GPU stored them (moe_backward's own deterministic
    # calls, repeated).
    dy_perm = moe.ops.unpermute_combine_bwd(bf(inp.dy), st.src_row)
    dgu, _, _ = moe.ops.grouped_gemm_down_bwd(dy_perm, st.h_w, st.gu_pre, st.w_perm, st.offsets, dn)
    moe.sync_status()
    xp, dg, hw, dyp = f64(st.x_perm), f64(dgu), f64(st.h_w), f64(dy_perm)
    offs = npi(st.offsets)
    own_gu, own_dn = np.zeros((E * H, 2 * I)), np.zeros((E * I, H))
    abs_gu, abs_dn = np.zeros((E * H, 2 * I)), np.zeros((E * I, H))
    for e in range(E):
        a, z = offs[e], offs[e + 1]
        own_gu[e * H:(e + 1) * H] = xp[a:z].T @ dg[a:z]
        own_dn[e * I:(e + 1) * I] = hw[a:z].T @ dyp[a:z]
        abs_gu[e * H:(e + 1) * H] = np.abs(xp[a:z]).T @ np.abs(dg[a:z])
        abs_dn[e * I:(e + 1) * I] = np.abs(hw[a:z]).T @ np.abs(dyp[a:z])
    assert_close("d_gate_up", f64(g["d_gate_up"]), b["d_gate_up"], operand_abs=abs_gu)
    assert_close("d_down", f64(g["d_down"]), b["d_down"], operand_abs=abs_dn)
    # and the two GEMMs themselves: the fp64 product of their stored operands,
    # within the bf16 store (half an ulp) and fp32 accumulation (2^-16 of
    # sum|a||b|, far below a bf16 ulp); a row of another expert leaking into
    # an expert's K tail would move an output by a whole product
    for name, got, own, ab in (("d_gate_up", g["d_gate_up"], own_gu, abs_gu), ("d_down", g["d_down"], own_dn, abs_dn)):
        err = np.abs(f64(got) - own)
        bound = bf16_allowance(own) - U_BF16 * np.abs(own) + 2.0 ** -16 * ab
        assert np.all(err <= bound), "%s vs its own operands: worst excess %.3g" % (name, (err - bound).max())


@pytest.mark.parametrize("T,H,E,k,I", _sweep_shapes(8, 777))
def test_seeded_shape_sweep_launch_variants_bit_identical(T, H, E, k, I):
    """At seeded irregular shapes, the forward (saving activations) and the
    backward give the same bits in every CTA-pair mode (single CTAs, pairs
    for the forward and dgrad GEMMs, pairs for gate_up and the
    weight-gradient GEMMs) and with the row gather fused into the gate_up
    load, as in the default launch (which the shape sweep above checks
    against the oracle)."""
    moe = lib()
    cfg, inp = _inputs(T, H, E, k, I, seed=T * 5 + E * 11 + k)
    variants = [(moe.GEMM_PAIRS_GATE_UP, "rows"), (moe.GEMM_PAIRS_NONE, "rows"), (moe.GEMM_PAIRS_ALL, "rows"),
                (moe.GEMM_PAIRS_GATE_UP_WGRAD, "rows"), (moe.GEMM_PAIRS_GATE_UP, "tma")]
    outs = []
    for pairs, fused in variants:
        moe.set_gemm_pairs(pairs)
        try:
            (x, wr, gu, dn), y, st = _forward(moe, inp, save=True, fused=fused)
            gr = moe.moe_backward(bf(inp.dy), st, wr, gu, dn, want_dw_router=True)
            moe.sync_status()
        finally:
            moe.set_gemm_pairs(moe.GEMM_PAIRS_GATE_UP)
        outs.append([y, st.ids, st.row_map, st.h, st.gu_pre, st.h_w, st.y_perm] + [gr[n] for n in sorted(gr)])
    for (pairs, fused), other in zip(variants[1:], outs[1:]):
        for i, (a, b) in enumerate(zip(outs[0], other)):
            assert torch_equal(a, b), "pairs mode %d, gather %s: output %d differs" % (pairs, fused, i)
