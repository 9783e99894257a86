"""Expert parallelism around the layer, emulated on one GPU.

The method wraps the expert layer in two all-to-alls ("Awesome-ML-SYS-Tutorial"
MoE/EP guide, gsyq.cn, "Expert Parallelism": dispatch, expert compute,
combine; LLaMA-Factory "FSDPTurbo EP/EFSDP" §3, the eager dispatcher).  Experts
are split over G ranks on dim 0 (rank d owns the experts [d E/G, (d+1) E/G)).
Per rank and step:

  1. route its own tokens, permute them by expert (rows are then grouped by
     destination rank) and gather the rows;
  2. exchange the per-(rank, expert) counts; a rank sends S[s][d] rows to
     rank d (the split sizes, read on the host as an all-to-all-v needs them);
  3. all-to-all of the rows: the rows of every sender go from (source,
     destination) chunk order to (destination, source) order;
  4. each receiver re-sorts its (source, local expert) chunks to (local
     expert, source) order (`sort_chunks_by_idxs`), runs the grouped GEMMs on
     its local experts, and sorts the results back;
  5. all-to-all back, and each source combines its rows with its gate weights.

This module runs the G ranks' steps one after the other on one device; the
two all-to-alls become the chunk transposes they are (moe_sort_chunks +
moe_permute_rows on the concatenated send buffers).  Everything else is the
library's single-device call a rank would make.  Since every expert then sees
its rows in the same order as the local layer (sources hold consecutive
token ranges), the output equals moe_forward's bit for bit, with or without
EPLB replicas, which is what the tests check.  A multi-GPU deployment replaces
the two transposes by an all-to-all-v of the same split sizes; this library
has no multi-GPU path of its own.

With fused_dispatch=True the receivers' gate_up GEMMs gather their A rows
straight from the senders' token rows (the grouped GEMM's TMA tile::gather4
load, through the composed index: receiver row -> (local expert, source) ->
the source's permuted row -> token), so neither the dispatch all-to-all nor
the re-sort copies a row: the data movement of an MC2-style fused
all-to-all + grouped GEMM ("FSDPTurbo EP/EFSDP" §3, the mc2 dispatcher; the
guide's DeepEP passage, compute starting as tokens arrive), on one device.
The composed index is built on the host from the sources' permutations.  On
GB300 the gathered load is slower than materialising the rows (it is bound
by the gather instruction rate), so it is off by default.

EPLB-style replication (the guide's hotspot experts): ``EPLBPlan`` gives hot
experts extra physical replicas (moe_eplb_plan, on the host) and spreads the
physical experts over the ranks; ``moe_ep_map_replicas`` sends each (token,
slot) of a replicated expert to replica token mod replicas.  The replicas'
weights are copies (``replicate_weights``).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import ops


@dataclass
class EPLBPlan:
    """Physical experts: phys_to_log [n_phys]; replica r of logical expert e is
    physical expert rep_list[rep_first[e] + r] (int32 numpy arrays, and their
    device copies ``*_dev``); rank g owns physical experts [g P, (g+1) P),
    P = n_phys / G; rank_load: the plan's load per rank."""
    G: int
    n_phys: int
    phys_to_log: np.ndarray
    rep_first: np.ndarray
    rep_count: np.ndarray
    rep_list: np.ndarray
    rank_load: np.ndarray
    rep_first_dev: torch.Tensor = None
    rep_count_dev: torch.Tensor = None
    rep_list_dev: torch.Tensor = None

    @staticmethod
    def build(expert_load, G, n_phys, device="cuda"):
        d = ops.eplb_plan(expert_load, G, n_phys)
        plan = EPLBPlan(G, n_phys, d["phys_to_log"], d["rep_first"], d["rep_count"], d["rep_list"],
                        d["rank_load"])
        if device is not None:
            plan.rep_first_dev = torch.from_numpy(plan.rep_first).to(device)
            plan.rep_count_dev = torch.from_numpy(plan.rep_count).to(device)
            plan.rep_list_dev = torch.from_numpy(plan.rep_list).to(device)
        return plan


def replicate_weights(gate_up, down, phys_to_log):
    """Physical expert weights [n_phys*H, 2I], [n_phys*I, H]: row blocks of the
    logical ones, copied by moe_permute_rows (a one-time weight preparation)."""
    n_phys = len(phys_to_log)
    E_H, twoI = gate_up.shape
    E_I, H = down.shape
    E = E_H // H
    I = E_I // E
    p2l = torch.from_numpy(np.asarray(phys_to_log, dtype=np.int64)).to(gate_up.device)
    rows_gu = (p2l[:, None] * H + torch.arange(H, device=gate_up.device)[None, :]).reshape(-1).to(torch.int32)
    rows_dn = (p2l[:, None] * I + torch.arange(I, device=gate_up.device)[None, :]).reshape(-1).to(torch.int32)
    return ops.permute_rows(gate_up, rows_gu), ops.permute_rows(down, rows_dn)


def token_ranges(T, G):
    """Consecutive token ranges of the G source ranks (the first T % G one longer)."""
    sizes = [T // G + (1 if s < T % G else 0) for s in range(G)]
    starts = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    return [(int(starts[s]), int(starts[s + 1])) for s in range(G)]


def ep_forward_emulated(x, w_router, gate_up, down, k, G, bias=None, plan: EPLBPlan | None = None,
                        phys_weights=None, stats=None, fused_dispatch=False):
    """The layer forward with experts split over G ranks, every rank's
    single-device steps run on this GPU in turn (see the module docstring).

    plan: an EPLBPlan (physical experts, replicas of hot experts) and
    phys_weights its (gate_up, down) from replicate_weights; without a plan
    the physical experts are the logical ones.  stats (a dict, optional)
    receives rows_per_rank [G] (the rows each rank's experts computed) and
    splits [G, G] (rows sent from source s to destination d).
    fused_dispatch: the receivers' gate_up GEMMs gather their rows from the
    senders' token rows (see the module docstring).
    Returns y [T, H] bf16, equal to moe_forward's bit for bit."""
    T, H = x.shape
    E = w_router.shape[1]
    I = down.shape[0] // E
    if plan is None:
        n_phys = E
        gu_p, dn_p = gate_up, down
    else:
        n_phys = plan.n_phys
        gu_p, dn_p = phys_weights if phys_weights is not None else replicate_weights(gate_up, down, plan.phys_to_log)
    if n_phys % G:
        raise ValueError("the physical experts (%d) must split evenly over %d ranks" % (n_phys, G))
    P = n_phys // G
    dev = x.device
    ranges = token_ranges(T, G)
    # 1. per source rank: route, map to replicas, permute, gather its rows
    src = []
    for (t0, t1) in ranges:
        xs = x[t0:t1]
        ids, w = ops.route(xs, w_router, k, bias)
        pids = ops.ep_map_replicas(ids, plan.rep_first_dev, plan.rep_count_dev, plan.rep_list_dev) \
            if plan is not None else ids
        counts, offsets, row_map, src_row = ops.permute(pids, n_phys)
        src.append(dict(x=xs, w=w, counts=counts, row_map=row_map, src_row=src_row))
    # 2. counts exchanged; split sizes on the host (as an all-to-all-v needs them)
    C_h = torch.stack([s["counts"] for s in src]).cpu().numpy().astype(np.int64)   # [G_src, n_phys]
    S = C_h.reshape(G, G, P).sum(2)                                # rows source s -> destination d
    n_send = S.sum(1)                                              # rows each source sends
    n_recv = S.sum(0)                                              # rows each destination receives
    N = int(S.sum())
    if stats is not None:
        stats["splits"] = S
        stats["rows_per_rank"] = n_recv
    base = np.concatenate([[0], np.cumsum(n_send)]).astype(np.int64)
    S_dev = torch.from_numpy(S.astype(np.int32)).to(dev)
    a2a_src, a2a_pos, _ = ops.sort_chunks(S_dev, N)
    if fused_dispatch:
        # the token of each row a receiver's experts see, in (local expert, source) order
        src_rows = [s["src_row"].cpu().numpy().astype(np.int64) for s in src]
        src_offs = [np.concatenate([[0], np.cumsum(C_h[s_i])]).astype(np.int64) for s_i in range(G)]
        t0s = [t0 for (t0, _) in ranges]
        recv = None
    else:
        # the send buffers side by side: every source gathers its rows into its slice
        send = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        for s_i, s in enumerate(src):
            ops.permute_rows(s["x"], s["src_row"], out=send[base[s_i]:base[s_i + 1]])
        # 3. all-to-all: (source, destination) chunks -> (destination, source)
        recv = ops.permute_rows(send, a2a_src)
    # 4. every destination: re-sort by local expert, grouped GEMMs, sort back
    y_recv = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
    rbase = np.concatenate([[0], np.cumsum(n_recv)]).astype(np.int64)
    for d in range(G):
        n_d = int(n_recv[d])
        if n_d == 0:
            continue
        # what rank d learns from the count exchange: [G_src, P] (source, local expert)
        recv_counts = torch.from_numpy(np.ascontiguousarray(C_h[:, d * P:(d + 1) * P]).astype(np.int32)).to(dev)
        s_src, s_pos, local_offsets = ops.sort_chunks(recv_counts, n_d)
        gu_d = gu_p[d * P * H:(d + 1) * P * H]
        dn_d = dn_p[d * P * I:(d + 1) * P * I]
        if fused_dispatch:
            tok = np.concatenate([src_rows[s_i][src_offs[s_i][d * P + e]:src_offs[s_i][d * P + e + 1]] + t0s[s_i]
                                  for e in range(P) for s_i in range(G)]).astype(np.int32)
            h, _, _ = ops.grouped_gemm_gate_up_swiglu(x, torch.from_numpy(tok).to(dev), local_offsets, gu_d, I)
        else:
            rows = ops.permute_rows(recv[rbase[d]:rbase[d] + n_d], s_src)
            h, _, _ = ops.grouped_gemm_gate_up_swiglu(rows, None, local_offsets, gu_d, I)
        y_sorted = ops.grouped_gemm_down(h, local_offsets, dn_d, H)
        ops.permute_rows(y_sorted, s_pos, out=y_recv[rbase[d]:rbase[d] + n_d])
    # 5. all-to-all back: (destination, source) -> (source, destination); combine
    y_send = ops.permute_rows(y_recv, a2a_pos)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    for s_i, (s, (t0, t1)) in enumerate(zip(src, ranges)):
        ops.unpermute_combine(y_send[base[s_i]:base[s_i + 1]], s["row_map"], s["w"], out=y[t0:t1])
    return y
