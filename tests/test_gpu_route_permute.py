"""GPU parity of the router, the permutation and the combine (through the C ABI)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import bf, f32, f64, i32, lib, npi
from parity import assert_close, compare_ids

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,H,E,k", [(64, 128, 8, 2), (1, 64, 4, 1), (333, 256, 16, 4), (1000, 512, 128, 8),
                                     (97, 128, 200, 8), (50, 64, 32, 32), (40, 96, 1024, 6),
                                     (129, 128, 48, 6), (257, 192, 240, 3), (300, 7168, 256, 8),
                                     (4100, 2048, 128, 8)])
def test_route_matches_oracle(T, H, E, k):
    """Shapes of the three router paths: the fused cluster kernel (16 <= E <=
    256, E % 16 == 0; clusters of 1 to 4 CTAs, 3 for E > 128, a partial 64-expert
    chunk, ragged 128-token tiles), the split-K tensor-core GEMM with a
    separate top-k (E % 8 == 0 otherwise) and the CUDA-core GEMM."""
    moe = lib()
    cfg = synth.MoEConfig("r", T=T, H=H, E=E, k=k, I=64, seed=T + E)
    inp = synth.make_inputs(cfg, weights=False)
    ids, w, logits = moe.route(bf(inp.x), f32(inp.w_router), k, return_logits=True)
    moe.sync_status()
    ref = oracle.route(inp.x, inp.w_router, None, k)
    same, tolerated = compare_ids(npi(ids), ref)
    assert tolerated <= max(1, T // 1000)
    assert_close("logits", f64(logits), ref["logits"], bf16_out=False)
    assert_close("w", f64(w)[same], ref["w"][same], bf16_out=False)
    np.testing.assert_allclose(f64(w).sum(1), 1.0, atol=1e-5)


@pytest.mark.parametrize("T,H,E,k,bias", [(4100, 2048, 128, 8, False), (333, 256, 16, 4, True),
                                          (97, 128, 200, 8, True), (40, 128, 1024, 6, False)])
def test_route_presplit_equals_route(T, H, E, k, bias):
    """W_r's split made once (moe_route_split_weight) and reused
    (moe_route_presplit) gives moe_route's ids, weights and logits bit for
    bit: on the fused cluster router (E = 128, 16) and the split-K path
    (E = 200, 1024); the split itself sums back to W_r exactly."""
    import torch
    moe = lib()
    cfg = synth.MoEConfig("r", T=T, H=H, E=E, k=k, I=64, seed=2 * T + E)
    inp = synth.make_inputs(cfg, weights=False)
    x, wr = bf(inp.x), f32(inp.w_router)
    b = f32(synth.zipf_bias(cfg.seed, E, 1.0)) if bias else None
    ref = moe.route(x, wr, k, b, return_logits=True)
    w_split = moe.route_split_weight(wr)
    for _ in range(2):   # the same split serves repeated calls
        got = moe.route(x, wr, k, b, return_logits=True, w_split=w_split)
        moe.sync_status()
        for a, c in zip(ref, got):
            assert torch.equal(a, c)
    parts = w_split.float().cpu().numpy().astype(np.float64).reshape(3, H, E)
    np.testing.assert_array_equal(parts.sum(0), inp.w_router.astype(np.float64))
    ids_ref = oracle.route(inp.x, inp.w_router, synth.zipf_bias(cfg.seed, E, 1.0) if bias else None, k)
    same, tolerated = compare_ids(npi(got[0]), ids_ref, label="presplit")
    assert tolerated <= max(1, T // 1000)


@pytest.mark.parametrize("H,E,k", [(2048, 128, 8), (7168, 256, 8), (256, 200, 6)])
def test_route_is_batch_invariant(H, E, k):
    """A token's logits, weights and experts do not depend on the tokens
    routed with it: slices of a batch (a single token, 511 tokens, an
    expert-parallel rank's share of 4096) routed alone give the same bits as
    the whole batch (the fused cluster router at E = 128 and 256, the split-K
    path at E = 200)."""
    import torch
    moe = lib()
    T = 4096
    cfg = synth.MoEConfig("r", T=T, H=H, E=E, k=k, I=64, seed=H + E)
    inp = synth.make_inputs(cfg, weights=False)
    x, wr = bf(inp.x), f32(inp.w_router)
    whole = moe.route(x, wr, k, return_logits=True)
    for t0, t1 in ((0, 1), (1000, 1511), (512, 1024), (3584, 4096)):
        part = moe.route(x[t0:t1].contiguous(), wr, k, return_logits=True)
        moe.sync_status()
        for a, b in zip(whole, part):
            assert torch.equal(a[t0:t1], b), (t0, t1)


def test_route_bias_and_skewed_workload():
    moe = lib()
    cfg = synth.CONFIGS["qwen3_moe_skewed"]
    inp = synth.make_inputs(cfg, weights=False)
    ids, w = moe.route(bf(inp.x), f32(inp.w_router), cfg.k, f32(inp.bias))
    moe.sync_status()
    ref = oracle.route(inp.x, inp.w_router, inp.bias, cfg.k)
    same, tolerated = compare_ids(npi(ids), ref)
    assert tolerated <= 4
    assert_close("w", f64(w)[same], ref["w"][same], bf16_out=False)
    counts = np.bincount(npi(ids).reshape(-1), minlength=cfg.E)
    assert (counts == 0).sum() >= 8 and counts.max() > 0.10 * cfg.R   # hotspot + empty experts


def test_route_exact_ties_lower_index_first():
    """Duplicate router columns give bit-identical fp32 logits on the GPU: the
    lower expert index must come first, and at the k boundary only it is kept."""
    moe = lib()
    T, H, E = 64, 128, 16
    rng = np.random.default_rng(0)
    xa = np.abs(synth.bf16_to_f32(synth.normal_bf16(3, synth.TID_X, (T, H), 1.0)))
    x = np.ascontiguousarray((xa.view(np.uint32) >> 16).astype(np.uint16))   # |x|, exact in bf16
    wr = (rng.standard_normal((H, E)) * 0.01).astype(np.float32)
    wr[:, 3] = 0.2     # experts 3 and 9 tie exactly and lead every token
    wr[:, 9] = 0.2
    wr[:, 12] = 0.1    # third
    for k, want in ((1, [3]), (2, [3, 9]), (3, [3, 9, 12])):
        ids, w = moe.route(bf(x), f32(wr), k)
        got = npi(ids)
        for t in range(T):
            assert got[t].tolist() == want
        if k >= 2:
            np.testing.assert_array_equal(npi(w)[:, 0], npi(w)[:, 1])


@pytest.mark.parametrize("T,k,E,kind", [(64, 2, 8, "distinct"), (1, 1, 1, "distinct"), (4096, 8, 128, "distinct"),
                                        (5000, 3, 7, "uniform"), (777, 8, 1024, "distinct"),
                                        (16384, 8, 256, "distinct"), (3000, 4, 64, "sparse"),
                                        (32768, 8, 256, "distinct"), (33000, 8, 128, "distinct"),
                                        (45000, 8, 128, "distinct")])
def test_permute_bit_exact(T, k, E, kind):
    """Every launch path of the permute: the cluster launch (R <= 2^18 and
    E <= 256; T = 32768, k = 8 is its largest size, 2048-assignment chunks),
    the one-launch cooperative permute (E = 1024; R = 264k), and (T = 45000,
    R = 360k: more 256-assignment blocks than fit on the device at once) the
    three-launch fallback."""
    moe = lib()
    if kind == "distinct":
        ids = synth.distinct_ids(T + k, synth.TID_IDS, T, k, E)
    elif kind == "uniform":
        ids = synth.uniform_ints(T, synth.TID_IDS, T * k, E).reshape(T, k)
    else:  # only a few experts used: many empty experts
        ids = (synth.uniform_ints(T, synth.TID_IDS, T * k, 5) * 7).astype(np.int32).reshape(T, k)
    counts, offsets, row_map, src_row = moe.permute(i32(ids), E)
    moe.sync_status()
    ref = oracle.permute(ids, E)
    np.testing.assert_array_equal(npi(counts), ref["counts"])
    np.testing.assert_array_equal(npi(offsets), ref["offsets"])
    np.testing.assert_array_equal(npi(row_map), ref["row_map"])
    np.testing.assert_array_equal(npi(src_row), ref["src_row"])


def test_permute_rejects_out_of_range_id_on_device():
    moe = lib()
    ids = np.array([[0, 1], [2, 9]], dtype=np.int32)
    moe.permute(i32(ids), 4)
    with pytest.raises(moe.MoEError) as ei:
        moe.sync_status()
    assert ei.value.status == 6   # MOE_ERR_DEVICE
    moe.sync_status()             # the status word was cleared


@pytest.mark.parametrize("T,H,k,shared", [(64, 128, 2, False), (300, 256, 8, True), (1, 64, 1, False),
                                          (1000, 2048, 8, False), (37, 136, 32, True), (3, 8, 4, True),
                                          (2000, 2056, 3, False), (5000, 2048, 8, False),
                                          (300, 7168, 8, True)])
def test_combine_matches_oracle(T, H, k, shared):
    """Shapes of the shared-memory gather: k = 32 with the shared expert's row
    (33 rows a stage), one 8-column chunk, a slice that is the whole odd-width
    row, many units per CTA (the stage ring wraps), and 896-column slices of
    7168-wide rows."""
    moe = lib()
    R = T * k
    yp_bits = synth.normal_bf16(5, 50, (R, H), 1.0)
    ys_bits = synth.normal_bf16(5, 51, (T, H), 1.0) if shared else None
    E = max(k, 16)
    ids = synth.distinct_ids(5, synth.TID_IDS, T, k, E)
    perm = oracle.permute(ids, E)
    _, _, row_map, _ = moe.permute(i32(ids), E)      # the GPU path's own permutation
    w = np.random.default_rng(T).uniform(0.05, 1.0, (T, k)).astype(np.float32)
    y = moe.unpermute_combine(bf(yp_bits), row_map, f32(w), bf(ys_bits) if shared else None)
    moe.sync_status()
    ref = oracle.unpermute_combine(synth.bf16_to_f32(yp_bits).astype(np.float64), perm["row_map"],
                                   w.astype(np.float64),
                                   synth.bf16_to_f32(ys_bits).astype(np.float64) if shared else None)
    assert_close("y", f64(y), ref)


@pytest.mark.parametrize("T,k,E,H", [(100, 4, 8, 256), (1, 1, 1, 8), (333, 8, 64, 1000), (50, 32, 40, 2056),
                                     (2049, 8, 128, 2048)])
def test_permute_rows_scatter_matches_oracle(T, k, E, H):
    """The token-by-token row move (each x row read once, written to its k
    permuted rows) against the oracle's row gather of the same permutation,
    bit for bit: H = 1000 and 2056 end inside a 1024-column slice; k = 32 is
    the largest k."""
    import torch
    moe = lib()
    ids = synth.distinct_ids(T + H, synth.TID_IDS, T, k, E)
    perm = oracle.permute(ids, E)
    _, _, row_map, _ = moe.permute(i32(ids), E)
    x = synth.normal_bf16(T + k, synth.TID_X, (T, H), 1.0)
    xp = moe.permute_rows_scatter(bf(x), row_map, k)
    moe.sync_status()
    np.testing.assert_array_equal(f64(xp), oracle.permute_rows(synth.bf16_to_f32(x), perm["src_row"]))


def test_permute_rows_scatter_reports_a_bad_destination():
    """A row_map entry outside [0, T*k) is reported (MOE_ERR_DEVICE) and that
    copy is not written; the other rows are."""
    import torch
    moe = lib()
    T, k, H = 16, 2, 64
    rm = torch.arange(T * k, dtype=torch.int32, device="cuda")
    rm[5] = T * k
    x = torch.ones((T, H), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((T * k, H), dtype=torch.bfloat16, device="cuda")
    moe.ops.call("moe_permute_rows_scatter", moe.ops._p(x), moe.ops._p(rm), T, k, H, moe.ops._p(out),
                 moe.ops._stream())
    with pytest.raises(moe.MoEError) as ei:
        moe.sync_status()
    assert ei.value.status == 6
    o = out.float().cpu().numpy()
    assert (o[5] == 0).all() and (np.delete(o, 5, axis=0) == 1).all()


def test_permute_rows_gathers():
    moe = lib()
    T, k, E, H = 100, 4, 8, 256
    ids = synth.distinct_ids(9, synth.TID_IDS, T, k, E)
    perm = oracle.permute(ids, E)
    _, _, _, src_row = moe.permute(i32(ids), E)
    x = synth.normal_bf16(9, synth.TID_X, (T, H), 1.0)
    xp = moe.permute_rows(bf(x), src_row)
    np.testing.assert_array_equal(npi(xp.view(__import__("torch").int16)).view(np.uint16), x[perm["src_row"]])
