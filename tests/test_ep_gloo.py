"""Expert-parallel dispatch and combine across real processes (gloo, world
sizes 2 and 4, CPU only), with the oracle's arithmetic.

Each rank holds 1/G of the tokens and of the experts (split on dim 0).
It routes its tokens, permutes them by expert, exchanges the per-expert
counts (all-gather), sends each rank its rows (all-to-all-v with the split
sizes from the counts), re-sorts the received chunks by local expert
(the oracle's sort_chunks, `sort_chunks_by_idxs` on the pages), computes its
experts, sorts the results back, returns them (all-to-all-v) and combines
("Awesome-ML-SYS-Tutorial" MoE/EP guide, gsyq.cn, "Expert Parallelism").
The gathered output must equal the single-process layer.  This checks the
host side of the exchange (split sizes, chunk orders) with a real
collective; no GPU is involved.
"""
import pytest
from test_bench_multirank import _run_ranks


@pytest.mark.parametrize("world", [2, 4])
def test_ep_dispatch_combine_across_ranks_equals_the_layer(world):
    """2 and 4 ranks (4 and 2 experts per rank; with 4 ranks a rank may
    receive nothing from some sources)."""
    outs = _run_ranks("""
        import numpy as np
        import torch
        import torch.distributed as dist
        import oracle
        import synth

        dist.init_process_group("gloo")
        rank, G = dist.get_rank(), dist.get_world_size()
        cfg = synth.MoEConfig("ep", T=64, H=128, E=8, k=2, I=64, seed=12)
        inp = synth.make_inputs(cfg)
        T, H, E, k, I = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I
        P = E // G
        t0, t1 = rank * T // G, (rank + 1) * T // G
        x = np.ascontiguousarray(inp.x[t0:t1])
        # 1. route and permute this rank's tokens
        r = oracle.route(x, inp.w_router, None, k)
        perm = oracle.permute(r["ids"], E)
        # 2. counts exchanged; split sizes
        counts = torch.from_numpy(perm["counts"].astype(np.int64))
        C = [torch.empty_like(counts) for _ in range(G)]
        dist.all_gather(C, counts)
        C = torch.stack(C).numpy()                          # [source, expert]
        S = C.reshape(G, G, P).sum(2)                       # rows source -> destination
        # 3. rows out (this rank's permuted rows are grouped by destination)
        send = torch.from_numpy(x[perm["src_row"]].astype(np.int32))
        recv = torch.empty((int(S[:, rank].sum()), H), dtype=torch.int32)
        dist.all_to_all_single(recv, send, output_split_sizes=S[:, rank].tolist(),
                               input_split_sizes=S[rank, :].tolist())
        # 4. re-sort (source, local expert) -> (local expert, source); the local experts
        src_of, pos_of, offs = oracle.sort_chunks(C[:, rank * P:(rank + 1) * P])
        rows = np.ascontiguousarray(recv.numpy().astype(np.uint16)[src_of])
        n = rows.shape[0]
        local = dict(counts=np.diff(offs).astype(np.int32), offsets=offs,
                     row_map=np.arange(n, dtype=np.int32), src_row=np.arange(n, dtype=np.int32))
        gu = np.ascontiguousarray(inp.gate_up[rank * P * H:(rank + 1) * P * H])
        dn = np.ascontiguousarray(inp.down[rank * P * I:(rank + 1) * P * I])
        _, extra = oracle.forward_permuted(rows, gu, dn, np.ones((n, 1)), local, 1, want_intermediates=True)
        y_recv = torch.from_numpy(np.ascontiguousarray(extra["y_perm"][pos_of]))
        # 5. rows back, combine
        y_perm = torch.empty((int(S[rank, :].sum()), H), dtype=torch.float64)
        dist.all_to_all_single(y_perm, y_recv, output_split_sizes=S[rank, :].tolist(),
                               input_split_sizes=S[:, rank].tolist())
        y = torch.from_numpy(oracle.unpermute_combine(y_perm.numpy(), perm["row_map"], r["w"]))
        ys = [torch.empty_like(y) for _ in range(G)]
        dist.all_gather(ys, y)
        if rank == 0:
            ref = oracle.layer_forward(inp)["y"]
            err = float(np.abs(torch.cat(ys).numpy() - ref).max())
            print("max err %.3g rows per rank %s" % (err, S.sum(0).tolist()))
            assert err < 1e-12
        dist.destroy_process_group()
    """, world=world)
    assert outs[0].startswith("max err")


@pytest.mark.parametrize("world", [2, 4])
def test_ep_with_eplb_replicas_across_ranks_equals_the_layer(world):
    """The same exchange over physical experts: the ranks sum their
    per-expert loads (all-reduce), plan 4 extra replicas of the busiest
    experts (the oracle's eplb_plan, hotspot experts and EPLB on the guide's
    "Expert Parallelism" page), send each assignment to replica t mod
    replicas of its expert (map_replicas) and hold the physical experts'
    copies of the logical weights.  The output is still the layer's."""
    outs = _run_ranks("""
        import numpy as np
        import torch
        import torch.distributed as dist
        import oracle
        import synth

        dist.init_process_group("gloo")
        rank, G = dist.get_rank(), dist.get_world_size()
        cfg = synth.MoEConfig("ep", T=64, H=128, E=8, k=2, I=64, seed=13)
        inp = synth.make_inputs(cfg)
        T, H, E, k, I = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I
        n_phys = E + 4
        P = n_phys // G
        t0, t1 = rank * T // G, (rank + 1) * T // G
        x = np.ascontiguousarray(inp.x[t0:t1])
        r = oracle.route(x, inp.w_router, None, k)
        # expert loads summed over the ranks, the plan, the physical experts
        load = torch.from_numpy(np.bincount(r["ids"].reshape(-1), minlength=E).astype(np.int64))
        dist.all_reduce(load)
        plan = oracle.eplb_plan(load.numpy(), G, n_phys)
        pids = oracle.map_replicas(r["ids"], plan["rep_first"], plan["rep_count"], plan["rep_list"])
        perm = oracle.permute(pids, n_phys)
        counts = torch.from_numpy(perm["counts"].astype(np.int64))
        C = [torch.empty_like(counts) for _ in range(G)]
        dist.all_gather(C, counts)
        C = torch.stack(C).numpy()
        S = C.reshape(G, G, P).sum(2)
        send = torch.from_numpy(x[perm["src_row"]].astype(np.int32))
        recv = torch.empty((int(S[:, rank].sum()), H), dtype=torch.int32)
        dist.all_to_all_single(recv, send, output_split_sizes=S[:, rank].tolist(),
                               input_split_sizes=S[rank, :].tolist())
        src_of, pos_of, offs = oracle.sort_chunks(C[:, rank * P:(rank + 1) * P])
        rows = np.ascontiguousarray(recv.numpy().astype(np.uint16)[src_of])
        n = rows.shape[0]
        local = dict(counts=np.diff(offs).astype(np.int32), offsets=offs,
                     row_map=np.arange(n, dtype=np.int32), src_row=np.arange(n, dtype=np.int32))
        mine = plan["phys_to_log"][rank * P:(rank + 1) * P]          # this rank's logical experts
        gu = np.ascontiguousarray(np.concatenate([inp.gate_up[e * H:(e + 1) * H] for e in mine]))
        dn = np.ascontiguousarray(np.concatenate([inp.down[e * I:(e + 1) * I] for e in mine]))
        _, extra = oracle.forward_permuted(rows, gu, dn, np.ones((n, 1)), local, 1, want_intermediates=True)
        y_recv = torch.from_numpy(np.ascontiguousarray(extra["y_perm"][pos_of]))
        y_perm = torch.empty((int(S[rank, :].sum()), H), dtype=torch.float64)
        dist.all_to_all_single(y_perm, y_recv, output_split_sizes=S[rank, :].tolist(),
                               input_split_sizes=S[:, rank].tolist())
        y = torch.from_numpy(oracle.unpermute_combine(y_perm.numpy(), perm["row_map"], r["w"]))
        ys = [torch.empty_like(y) for _ in range(G)]
        dist.all_gather(ys, y)
        if rank == 0:
            ref = oracle.layer_forward(inp)["y"]
            err = float(np.abs(torch.cat(ys).numpy() - ref).max())
            print("max err %.3g replicas %s rows per rank %s" % (err, plan["rep_count"].tolist(),
                                                                S.sum(0).tolist()))
            assert err < 1e-12
            assert plan["rep_count"].sum() == n_phys and plan["rep_count"].max() > 1
        dist.destroy_process_group()
    """, world=world)
    assert outs[0].startswith("max err")
