"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test names what it pins.  The oracle restates the pages' definitions:
router (gate -> FP32 softmax -> top-k -> renormalise) and experts
(permute -> grouped matmul -> SwiGLU -> grouped matmul -> unpermute) from
"InternVL3.5 接入 pure FSDP2 后端开发实践" (MindSpeed-MM issue 625) §2, §8.2,
§8.3, and the plain MoE forward of the Awesome-ML-SYS-Tutorial MoE/EP guide
(gsyq.cn), "Expert Parallelism".
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f64(bits):
    return synth.bf16_to_f32(bits).astype(np.float64)


def _tiny(seed=0, T=64, H=128, E=8, k=2, I=64):
    cfg = synth.MoEConfig("t", T=T, H=H, E=E, k=k, I=I, seed=seed)
    return synth.make_inputs(cfg, with_dy=True)


def _rand_f64(rng, shape, scale=1.0):
    return np.ascontiguousarray(rng.standard_normal(shape) * scale)


# ---------------------------------------------------------------- router pins

def test_route_matches_sort_based_topk():
    """Pin: an independent top-k (numpy softmax via scipy + lexsort on
    (-p, index)) on numpy-matmul logits gives the same ids and weights."""
    inp = _tiny(seed=0)
    r = oracle.route(inp.x, inp.w_router, None, 2)
    z = _f64(inp.x) @ inp.w_router.astype(np.float64)
    p = scipy.special.softmax(z, axis=1)
    T, E = p.shape
    for t in range(T):
        order = np.lexsort((np.arange(E), -p[t]))[:2]
        assert r["kgap"][t] > 1e-9, "a near tie would make this comparison ill-posed"
        np.testing.assert_array_equal(r["ids"][t], order)
        np.testing.assert_allclose(r["w"][t], p[t, order] / p[t, order].sum(), rtol=1e-12)
    np.testing.assert_allclose(r["logits"], z, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["probs"], p, rtol=1e-12, atol=1e-15)


def test_route_with_bias_matches_sort_based_topk():
    """Pin: the bias enters the logits before the softmax (same brute force)."""
    inp = _tiny(seed=5, T=32, E=16, k=4)
    bias = synth.zipf_bias(5, 16, 1.0)
    r = oracle.route(inp.x, inp.w_router, bias, 4)
    z = _f64(inp.x) @ inp.w_router.astype(np.float64) + bias.astype(np.float64)
    p = scipy.special.softmax(z, axis=1)
    for t in range(32):
        order = np.lexsort((np.arange(16), -p[t]))[:4]
        np.testing.assert_array_equal(r["ids"][t], order)
        np.testing.assert_allclose(r["w"][t], p[t, order] / p[t, order].sum(), rtol=1e-12)


def test_route_exact_ties_go_to_lower_index():
    """Pin: duplicated router columns give bit-identical logits; the lower
    expert index must come first, and at the k boundary only it is chosen."""
    rng = np.random.default_rng(1)
    T, H, E = 16, 32, 8
    x = _rand_f64(rng, (T, H))
    w_r = _rand_f64(rng, (H, E), 0.1)
    # experts 2 and 6 share a column scaled up so that they lead every token
    lead = np.sign(x.sum(1, keepdims=True)).T  # not needed per token: build per token below
    del lead
    col = np.ascontiguousarray(x.mean(0) * 50.0)
    w_r[:, 2] = col
    w_r[:, 6] = col
    w_r[:, 5] = col * 0.5  # third
    xs = np.ascontiguousarray(np.abs(x) * np.sign(col)[None, :])  # make x . col > 0
    r2 = oracle.route(xs, w_r, None, 2)
    r3 = oracle.route(xs, w_r, None, 3)
    r1 = oracle.route(xs, w_r, None, 1)
    for t in range(T):
        assert r2["logits"][t, 2] == r2["logits"][t, 6]
        np.testing.assert_array_equal(r2["ids"][t], [2, 6])
        np.testing.assert_array_equal(r3["ids"][t], [2, 6, 5])
        np.testing.assert_array_equal(r1["ids"][t], [2])      # tie at the boundary
        assert r2["w"][t, 0] == r2["w"][t, 1] == 0.5


def test_route_weights_sum_to_one_and_equal_selected_softmax():
    """Invariants: w sums to 1 per token; renormalised softmax equals the
    softmax over the chosen logits alone; weights are non-increasing."""
    inp = _tiny(seed=2, E=16, k=4)
    r = oracle.route(inp.x, inp.w_router, None, 4)
    np.testing.assert_allclose(r["w"].sum(1), 1.0, rtol=0, atol=1e-12)
    zsel = np.take_along_axis(r["logits"], r["ids"].astype(np.int64), axis=1)
    np.testing.assert_allclose(r["w"], scipy.special.softmax(zsel, axis=1), rtol=1e-12)
    assert np.all(np.diff(r["w"], axis=1) <= 1e-15)


def test_route_k_equals_E_gives_softmax():
    """Special case: k == E selects everything, so w equals the softmax."""
    inp = _tiny(seed=3, E=8, k=8)
    r = oracle.route(inp.x, inp.w_router, None, 8)
    p = scipy.special.softmax(_f64(inp.x) @ inp.w_router.astype(np.float64), axis=1)
    for t in range(inp.x.shape[0]):
        np.testing.assert_allclose(r["w"][t], p[t, r["ids"][t]], rtol=1e-12)
        assert sorted(r["ids"][t].tolist()) == list(range(8))
    assert np.all(np.isinf(r["kgap"]))


def test_weights_for_ids_matches_router_and_probabilities():
    """Pin of weights_for_ids (the renormalised weights of a given choice):
    on the router's own choice it equals the C router's w; on any other
    choice (a permuted, reordered and arbitrary set) it equals p_e / sum p
    from the brute-force scipy softmax over all E experts."""
    inp = _tiny(seed=4, E=16, k=4)
    r = oracle.route(inp.x, inp.w_router, None, 4)
    np.testing.assert_allclose(oracle.weights_for_ids(r["logits"], r["ids"]), r["w"], rtol=1e-13)
    p = scipy.special.softmax(_f64(inp.x) @ inp.w_router.astype(np.float64), axis=1)
    rng = np.random.default_rng(4)
    other = np.stack([rng.permutation(16)[:4] for _ in range(p.shape[0])]).astype(np.int32)
    want = np.take_along_axis(p, other.astype(np.int64), axis=1)
    want /= want.sum(1, keepdims=True)
    np.testing.assert_allclose(oracle.weights_for_ids(r["logits"], other), want, rtol=1e-12)


# --------------------------------------------------------------- permute pins

def _check_perm(ids, E, perm):
    T, k = ids.shape
    R = T * k
    flat = ids.reshape(-1)
    c, off, rm, sr = perm["counts"], perm["offsets"], perm["row_map"], perm["src_row"]
    assert c.sum() == R
    np.testing.assert_array_equal(c, np.bincount(flat, minlength=E))
    assert off[0] == 0 and off[E] == R
    np.testing.assert_array_equal(np.diff(off), c)
    assert sorted(rm.tolist()) == list(range(R))               # a permutation
    np.testing.assert_array_equal(sr[rm], np.arange(R) // k)   # src_row inverts it on tokens
    for i in range(R):                                         # rows land in their expert's range
        assert off[flat[i]] <= rm[i] < off[flat[i] + 1]
    # stability by brute force: a stable sort of i by expert lists the rows in order
    order = sorted(range(R), key=lambda i: (flat[i], i))
    np.testing.assert_array_equal(rm[np.array(order)], np.arange(R))


@pytest.mark.parametrize("T,k,E", [(64, 2, 8), (37, 3, 5), (1, 1, 1), (16, 4, 4), (100, 8, 128)])
def test_permute_invariants_and_stability(T, k, E):
    ids = synth.distinct_ids(11, synth.TID_IDS, T, k, E)
    _check_perm(ids, E, oracle.permute(ids, E))


def test_permute_with_repeats_and_empty_experts():
    """Empty experts are legal (FSDPTurbo EP/EFSDP design notes, dispatcher
    table: fused path with empty experts); two experts never chosen."""
    T, k, E = 50, 2, 8
    ids = synth.uniform_ints(7, synth.TID_IDS, T * k, 6).reshape(T, k)  # experts 6, 7 empty
    perm = oracle.permute(ids, E)
    _check_perm(ids, E, perm)
    assert perm["counts"][6] == 0 and perm["counts"][7] == 0
    assert perm["offsets"][6] == perm["offsets"][7] == perm["offsets"][8] == T * k


def test_permute_rejects_out_of_range():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 3]], np.int32), 3)


def test_permute_unpermute_round_trip_is_identity():
    """Pin: permuting rows and combining them back with weights summing to 1
    (w = 1/k; k a power of two, so exact) returns x bit for bit; arbitrary
    weights return (sum_j w[t,j]) * x[t]."""
    inp = _tiny(seed=4, T=48, E=8, k=4)
    x = _f64(inp.x)
    ids = synth.distinct_ids(4, synth.TID_IDS, 48, 4, 8)
    perm = oracle.permute(ids, 8)
    xp = oracle.permute_rows(x, perm["src_row"])
    y = oracle.unpermute_combine(xp, perm["row_map"], np.full((48, 4), 0.25))
    np.testing.assert_array_equal(y, x)
    w = np.random.default_rng(0).uniform(0.1, 1.0, (48, 4))
    y2 = oracle.unpermute_combine(xp, perm["row_map"], w)
    np.testing.assert_allclose(y2, w.sum(1, keepdims=True) * x, rtol=1e-14)


# --------------------------------------------------------------- forward pins

def test_hand_case_closed_form():
    """Pin: a hand-computable layer (tests/golden/swiglu_hand_case.json) with
    H=2, I=1, E=2; expected values are closed forms of the definition."""
    with open(os.path.join(GOLDEN, "swiglu_hand_case.json")) as f:
        g = json.load(f)
    x = np.array(g["x"], dtype=np.float64)
    w_r = np.array(g["w_r"], dtype=np.float64)
    gu = np.array(g["gate_up"], dtype=np.float64)
    dn = np.array(g["down"], dtype=np.float64)
    silu = lambda v: v / (1.0 + math.exp(-v))
    # token 0: z = (2, -0.5); expert 0: g = 1, u = 2; expert 1: g = 0.5, u = 3
    f00 = silu(1.0) * 2.0 * np.array([2.0, -1.0])
    f01 = silu(0.5) * 3.0 * np.array([0.5, 3.0])
    # token 1: z = (-0.75, 1.125); expert 1: g = 1.375, u = -1.75; expert 0: g = -0.375, u = -0.75
    f11 = silu(1.375) * -1.75 * np.array([0.5, 3.0])
    f10 = silu(-0.375) * -0.75 * np.array([2.0, -1.0])
    r1 = oracle.route(x, w_r, None, 1)
    np.testing.assert_array_equal(r1["ids"], [[0], [1]])
    np.testing.assert_allclose(r1["logits"], [[2.0, -0.5], [-0.75, 1.125]], rtol=0, atol=1e-15)
    y1 = oracle.forward_permuted(x, gu, dn, r1["w"], oracle.permute(r1["ids"], 2), 1)
    np.testing.assert_allclose(y1, [f00, f11], rtol=1e-14)
    r2 = oracle.route(x, w_r, None, 2)
    np.testing.assert_array_equal(r2["ids"], [[0, 1], [1, 0]])
    a0 = 1.0 / (1.0 + math.exp(-2.5))
    a1 = 1.0 / (1.0 + math.exp(-1.875))
    np.testing.assert_allclose(r2["w"], [[a0, 1 - a0], [a1, 1 - a1]], rtol=1e-14)
    y2 = oracle.forward_permuted(x, gu, dn, r2["w"], oracle.permute(r2["ids"], 2), 2)
    np.testing.assert_allclose(y2, [a0 * f00 + (1 - a0) * f01, a1 * f11 + (1 - a1) * f10], rtol=1e-14)


def test_permuted_equals_bruteforce_dense():
    """Pin: the permuted form (histogram, scan, stable scatter, per-expert
    loops, gather-combine) equals computing every expert on every token and
    masking by the routing."""
    inp = _tiny(seed=0)
    r = oracle.route(inp.x, inp.w_router, None, 2)
    perm = oracle.permute(r["ids"], 8)
    y = oracle.forward_permuted(inp.x, inp.gate_up, inp.down, r["w"], perm, 2)
    yd = oracle.forward_dense(inp.x, inp.gate_up, inp.down, r["ids"], r["w"])
    np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-12 * np.abs(yd).max())
    yt = oracle.forward_tokens(np.arange(64), inp.x, inp.gate_up, inp.down, r["ids"], r["w"])
    np.testing.assert_allclose(yt, yd, rtol=1e-12, atol=1e-12 * np.abs(yd).max())


@pytest.mark.parametrize("skew,I_s", [(False, 0), (True, 0), (False, 32)])
def test_layer_forward_equals_per_token_definition(skew, I_s):
    """Pin of the composition: layer_forward (route -> permute -> permuted
    experts -> combine, with the router bias of a skewed config and a shared
    expert) equals the per-token definition computed by brute force: every
    expert on every token, masked by the routing the bias produces, plus the
    shared FFN on every token."""
    cfg = synth.MoEConfig("pin", T=48, H=64, E=6, k=2, I=32, seed=5, skew=skew, I_shared=I_s)
    inp = synth.make_inputs(cfg, bias_scale=1.0 if skew else None)
    res = oracle.layer_forward(inp)
    r = oracle.route(inp.x, inp.w_router, inp.bias, cfg.k)
    np.testing.assert_array_equal(res["route"]["ids"], r["ids"])
    yd = oracle.forward_dense(inp.x, inp.gate_up, inp.down, r["ids"], r["w"], inp.sh_gate_up, inp.sh_down)
    np.testing.assert_allclose(res["y"], yd, rtol=1e-12, atol=1e-12 * np.abs(yd).max())
    if skew:
        assert inp.bias is not None and not np.array_equal(
            r["ids"], oracle.route(inp.x, inp.w_router, None, cfg.k)["ids"])   # the bias changes the routing
    if I_s:
        y_no_shared = oracle.forward_dense(inp.x, inp.gate_up, inp.down, r["ids"], r["w"])
        assert np.abs(res["y"] - y_no_shared).max() > 1e-3                     # the shared expert is added


def test_dense_ffn_matches_library_matmul():
    """Pin: the SwiGLU FFN against numpy matmuls (library routine), which also
    fixes gate = first I columns, up = last I columns, and operand orientation."""
    rng = np.random.default_rng(3)
    T, H, I = 9, 24, 10
    x, gu, dn = _rand_f64(rng, (T, H)), _rand_f64(rng, (H, 2 * I), 0.3), _rand_f64(rng, (I, H), 0.3)
    g, u = x @ gu[:, :I], x @ gu[:, I:]
    ref = (g * scipy.special.expit(g) * u) @ dn
    np.testing.assert_allclose(oracle.dense_ffn(x, gu, dn), ref, rtol=1e-12, atol=1e-13)


def test_identical_experts_reduce_to_one_dense_ffn():
    """Pin: with every expert given the same weights the renormalised gate
    weights sum to 1, so the layer equals one dense SwiGLU FFN."""
    inp = _tiny(seed=6, T=40, E=8, k=3)
    H, I, E = 128, 64, 8
    gu = np.ascontiguousarray(np.tile(inp.gate_up[:H], (E, 1)))
    dn = np.ascontiguousarray(np.tile(inp.down[:I], (E, 1)))
    r = oracle.route(inp.x, inp.w_router, None, 3)
    y = oracle.forward_permuted(inp.x, gu, dn, r["w"], oracle.permute(r["ids"], E), 3)
    yref = oracle.dense_ffn(inp.x, inp.gate_up[:H], inp.down[:I])
    np.testing.assert_allclose(y, yref, rtol=1e-12, atol=1e-12 * np.abs(yref).max())


def test_shared_expert_adds_one_dense_ffn():
    """Pin: the always-active shared expert adds exactly one dense SwiGLU FFN
    of x with weight 1 (Awesome-ML-SYS-Tutorial MoE/EP guide: shared experts)."""
    cfg = synth.MoEConfig("s", T=24, H=64, E=4, k=2, I=32, seed=9, I_shared=48)
    inp = synth.make_inputs(cfg)
    r = oracle.route(inp.x, inp.w_router, None, 2)
    perm = oracle.permute(r["ids"], 4)
    y0 = oracle.forward_permuted(inp.x, inp.gate_up, inp.down, r["w"], perm, 2)
    y1, ex = oracle.forward_permuted(inp.x, inp.gate_up, inp.down, r["w"], perm, 2, inp.sh_gate_up,
                                     inp.sh_down, want_intermediates=True)
    ys = oracle.dense_ffn(inp.x, inp.sh_gate_up, inp.sh_down)
    np.testing.assert_allclose(y1 - y0, ys, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(ex["y_shared"], ys, rtol=0, atol=0)
    yd = oracle.forward_dense(inp.x, inp.gate_up, inp.down, r["ids"], r["w"], inp.sh_gate_up, inp.sh_down)
    np.testing.assert_allclose(y1, yd, rtol=1e-12, atol=1e-12 * np.abs(yd).max())


def test_intermediates_consistent():
    """The saved intermediates satisfy their definitions: h = silu(g) * u and
    y = sum_j w * y_perm[row_map]."""
    inp = _tiny(seed=8)
    r = oracle.route(inp.x, inp.w_router, None, 2)
    perm = oracle.permute(r["ids"], 8)
    y, ex = oracle.forward_permuted(inp.x, inp.gate_up, inp.down, r["w"], perm, 2, want_intermediates=True)
    g, u = ex["gu_perm"][:, :64], ex["gu_perm"][:, 64:]
    np.testing.assert_allclose(ex["h_perm"], g * scipy.special.expit(g) * u, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(oracle.unpermute_combine(ex["y_perm"], perm["row_map"], r["w"]), y, rtol=1e-14)


# -------------------------------------------------------------- backward pins

def _fd_problem(seed=0, T=3, H=6, E=4, k=2, I=5):
    rng = np.random.default_rng(seed)
    while True:
        x = _rand_f64(rng, (T, H))
        w_r = _rand_f64(rng, (H, E), 1.0 / math.sqrt(H))
        gu = _rand_f64(rng, (E * H, 2 * I), 1.0 / math.sqrt(H))
        dn = _rand_f64(rng, (E * I, H), 1.0 / math.sqrt(I))
        dy = _rand_f64(rng, (T, H))
        r = oracle.route(x, w_r, None, k)
        if r["kgap"].min() > 0.05:  # far from any routing flip under a 1e-6 perturbation
            return x, w_r, gu, dn, dy, k


def _loss(x, w_r, gu, dn, dy, k, bias=None):
    r = oracle.route(x, w_r, bias, k)
    y = oracle.forward_permuted(x, gu, dn, r["w"], oracle.permute(r["ids"], w_r.shape[1]), k)
    return float((dy * y).sum())


def _fd_check(fn, arr, grad, n_coords=12, seed=0, delta=1e-6):
    rng = np.random.default_rng(seed)
    flat = arr.reshape(-1)
    idx = rng.choice(flat.size, size=min(n_coords, flat.size), replace=False)
    fd = []
    for i in idx:
        old = flat[i]
        flat[i] = old + delta
        lp = fn()
        flat[i] = old - delta
        lm = fn()
        flat[i] = old
        fd.append((lp - lm) / (2 * delta))
    fd = np.array(fd)
    an = grad.reshape(-1)[idx]
    err = np.linalg.norm(fd - an) / max(np.linalg.norm(an), 1e-300)
    assert err < 1e-6, (err, fd, an)


def test_backward_matches_finite_differences():
    """Pin: central finite differences of the fp64 forward (routing recomputed,
    far from any top-k boundary) match the analytic dX, d_gate_up, d_down,
    d_w_r and (through a per-expert bias) d_logits."""
    x, w_r, gu, dn, dy, k = _fd_problem()
    r = oracle.route(x, w_r, None, k)
    b = oracle.backward(x, w_r, gu, dn, r["ids"], r["w"], dy, want_dw=True, want_dwr=True)
    L = lambda: _loss(x, w_r, gu, dn, dy, k)
    _fd_check(L, x, b["dX"], n_coords=18)
    _fd_check(L, gu, b["d_gate_up"], n_coords=40, seed=1)
    _fd_check(L, dn, b["d_down"], n_coords=40, seed=2)
    _fd_check(L, w_r, b["d_w_r"], n_coords=20, seed=3)
    bias = np.zeros(w_r.shape[1])
    _fd_check(lambda: _loss(x, w_r, gu, dn, dy, k, bias), bias, b["dlogits"].sum(0), n_coords=4, seed=4)


def test_backward_logit_grad_per_token_matches_fd():
    """Pin: per token, d_logits equals the finite-difference gradient with
    respect to that token's logits (a bias perturbation with T = 1)."""
    x, w_r, gu, dn, dy, k = _fd_problem(seed=5, T=1, E=6, k=3)
    r = oracle.route(x, w_r, None, k)
    b = oracle.backward(x, w_r, gu, dn, r["ids"], r["w"], dy, want_dw=False)
    bias = np.zeros(w_r.shape[1])
    _fd_check(lambda: _loss(x, w_r, gu, dn, dy, k, bias), bias, b["dlogits"][0], n_coords=6)
    unchosen = np.setdiff1d(np.arange(6), r["ids"][0])
    assert np.all(b["dlogits"][0, unchosen] == 0.0)


def test_logit_grad_sums_to_zero():
    """Invariant: softmax gradients sum to zero over the experts of a token."""
    inp = _tiny(seed=12, T=32, E=8, k=3)
    r = oracle.route(inp.x, inp.w_router, None, 3)
    b = oracle.backward(inp.x, inp.w_router, inp.gate_up, inp.down, r["ids"], r["w"], inp.dy,
                        want_dw=False)
    scale = np.abs(b["dlogits"]).max()
    np.testing.assert_allclose(b["dlogits"].sum(1), 0.0, atol=1e-13 * scale)


def test_sampled_backward_matches_full():
    """The token-sampled and expert-sampled backward equal the full one."""
    inp = _tiny(seed=13, T=40, E=8, k=2)
    r = oracle.route(inp.x, inp.w_router, None, 2)
    full = oracle.backward(inp.x, inp.w_router, inp.gate_up, inp.down, r["ids"], r["w"], inp.dy)
    tok = np.array([0, 7, 39, 12])
    bt = oracle.backward_tokens(tok, inp.x, inp.w_router, inp.gate_up, inp.down, r["ids"], r["w"], inp.dy)
    np.testing.assert_allclose(bt["dX"], full["dX"][tok], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(bt["dlogits"], full["dlogits"][tok], rtol=1e-13, atol=1e-15)
    for e in (0, 5):
        dgu, ddn = oracle.backward_expert(e, inp.x, inp.gate_up, inp.down, r["ids"], r["w"], inp.dy)
        np.testing.assert_array_equal(dgu, full["d_gate_up"][e * 128:(e + 1) * 128])
        np.testing.assert_array_equal(ddn, full["d_down"][e * 64:(e + 1) * 64])


def test_backward_empty_expert_has_zero_weight_grad():
    """An expert no token chose gets a zero weight gradient."""
    inp = _tiny(seed=14, T=16, E=8, k=2)
    ids = synth.uniform_ints(3, synth.TID_IDS, 32, 7).reshape(16, 2)  # expert 7 empty
    ids[:, 1] = np.where(ids[:, 1] == ids[:, 0], (ids[:, 0] + 1) % 7, ids[:, 1])
    w = np.full((16, 2), 0.5)
    dgu, ddn = oracle.backward_expert(7, inp.x, inp.gate_up, inp.down, ids, w, inp.dy)
    assert not dgu.any() and not ddn.any()
