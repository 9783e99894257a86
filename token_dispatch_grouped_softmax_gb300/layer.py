"""The MoE expert layer as a sequence of library calls, plus a torch autograd
Function around it.

Forward ("InternVL3.5 接入 pure FSDP2 后端开发实践", MindSpeed-MM issue 625,
§8.2-§8.3): route -> permute -> grouped gate_up GEMM + SwiGLU -> grouped down
GEMM -> unpermute-combine (+ the shared expert, "Awesome-ML-SYS-Tutorial"
MoE/EP guide: shared experts are always active).  All calls are enqueued on
the current stream with no host synchronisation: expert_offsets stay on the
device and the grouped GEMMs read them there.

Backward: combine_bwd (dY rows to permuted order) -> down_bwd -> route_bwd ->
gate_up_bwd -> gather_dx.
"""
from __future__ import annotations

import contextlib
from dataclasses import dataclass

import torch

from . import ops


def _range(name):
    """An NVTX range around one step of the layer, so that a profiler's
    timeline (Nsight Systems, Nsight Compute's NVTX filters) shows which
    library call enqueued each kernel; inside a CUDA graph capture the ranges
    mark the capture only."""
    nvtx = getattr(torch.cuda, "nvtx", None)
    return nvtx.range(name) if nvtx is not None else contextlib.nullcontext()


@dataclass
class ForwardState:
    """What the forward keeps for the backward."""
    x: torch.Tensor
    ids: torch.Tensor
    w: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    row_map: torch.Tensor
    src_row: torch.Tensor
    h: torch.Tensor
    y_perm: torch.Tensor
    w_perm: torch.Tensor | None = None
    gu_pre: torch.Tensor | None = None     # fp32 [R, 2I]
    h_w: torch.Tensor | None = None        # bf16 w * h [R, I]
    x_perm: torch.Tensor | None = None     # bf16 [R, H] when the rows were materialised
    y_shared: torch.Tensor | None = None


def moe_forward(x, w_router, gate_up, down, k, bias=None, sh_gate_up=None, sh_down=None,
                save_for_backward=False, fused_gather=False, w_split=None):
    """y [T, H] bf16 and the ForwardState.

    fused_gather: the grouped gate_up GEMM gathers the token rows itself (the
    permute fused into the operand load by TMA tile::gather4); False
    (default) materialises the permuted rows first (moe_permute_rows_scatter) and
    streams them with 128-row TMA tiles, which measures ~2.5x faster for the
    GEMM on GB300.
    w_split: W_r's bf16 split (ops.route_split_weight), prepared once while
    W_r does not change; the same results as without it."""
    T, H = x.shape
    E = w_router.shape[1]
    I = down.shape[0] // E
    with _range("moe.route"):
        ids, w = ops.route(x, w_router, k, bias, w_split=w_split)
    w_perm = None
    with _range("moe.permute"):
        if save_for_backward:
            counts, offsets, row_map, src_row, w_perm = ops.permute(ids, E, w)
        else:
            counts, offsets, row_map, src_row = ops.permute(ids, E)
    x_perm = None
    if fused_gather:
        with _range("moe.gate_up"):
            h, gu_pre, h_w = ops.grouped_gemm_gate_up_swiglu(x, src_row, offsets, gate_up, I, w_perm=w_perm,
                                                             save_for_backward=save_for_backward)
    else:
        with _range("moe.permute_rows"):
            x_perm = ops.permute_rows_scatter(x, row_map, k)
        with _range("moe.gate_up"):
            h, gu_pre, h_w = ops.grouped_gemm_gate_up_swiglu(x_perm, None, offsets, gate_up, I, w_perm=w_perm,
                                                             save_for_backward=save_for_backward)
    with _range("moe.down"):
        y_perm = ops.grouped_gemm_down(h, offsets, down, H)
    y_shared = None
    if sh_gate_up is not None:
        I_s = sh_down.shape[0]
        with _range("moe.shared_expert"):
            hs, _, _ = ops.grouped_gemm_gate_up_swiglu(x, None, None, sh_gate_up, I_s)
            y_shared = ops.grouped_gemm_down(hs, None, sh_down, H)
    with _range("moe.combine"):
        y = ops.unpermute_combine(y_perm, row_map, w, y_shared)
    st = ForwardState(x, ids, w, counts, offsets, row_map, src_row, h, y_perm, w_perm, gu_pre, h_w, x_perm,
                      y_shared)
    return y, st


def moe_backward(dy, st: ForwardState, w_router, gate_up, down, want_dw_router=False):
    """dict(dx, d_logits, d_gate_up, d_down, dw[, d_w_router]) for upstream gradient dy."""
    if st.gu_pre is None:
        raise ValueError("the forward ran without save_for_backward=True")
    T, H = st.x.shape
    E = w_router.shape[1]
    k = st.w.shape[1]
    with _range("moe.combine_bwd"):
        # dy_perm[row] = dY[src_row[row]], moved token by token (each dY row read
        # once; the same bits as ops.unpermute_combine_bwd, the gather)
        dy_perm = ops.permute_rows_scatter(dy, st.row_map, k)
    with _range("moe.down_bwd"):
        dgu, d_down, dw_part = ops.grouped_gemm_down_bwd(dy_perm, st.h_w, st.gu_pre, st.w_perm, st.offsets, down)
    with _range("moe.route_bwd"):
        d_logits, dw = ops.route_bwd(dw_part, st.row_map, st.w, st.ids, E)
    with _range("moe.gate_up_bwd"):
        if st.x_perm is not None:
            dx_perm, d_gate_up = ops.grouped_gemm_gate_up_bwd(dgu, st.x_perm, None, st.offsets, gate_up)
        else:
            dx_perm, d_gate_up = ops.grouped_gemm_gate_up_bwd(dgu, st.x, st.src_row, st.offsets, gate_up)
    with _range("moe.gather_dx"):
        dx = ops.gather_dx(dx_perm, st.row_map, T, k, d_logits, st.ids, w_router)
    out = dict(dx=dx, d_logits=d_logits, d_gate_up=d_gate_up, d_down=d_down, dw=dw)
    if want_dw_router:
        with _range("moe.route_bwd_weight"):
            out["d_w_router"] = ops.route_bwd_weight(st.x, d_logits)
    return out


class MoELayerFunction(torch.autograd.Function):
    """y = MoE(x); gradients for x, W_r, gate_up and down (fp32 W_r grad)."""

    @staticmethod
    def forward(ctx, x, w_router, gate_up, down, k, bias):
        y, st = moe_forward(x.contiguous(), w_router.contiguous(), gate_up.contiguous(),
                            down.contiguous(), k, bias, save_for_backward=True)
        ctx.st = st
        ctx.save_for_backward(w_router, gate_up, down)
        return y

    @staticmethod
    def backward(ctx, dy):
        w_router, gate_up, down = ctx.saved_tensors
        g = moe_backward(dy.contiguous(), ctx.st, w_router, gate_up, down,
                         want_dw_router=ctx.needs_input_grad[1])
        return (g["dx"], g.get("d_w_router"), g["d_gate_up"], g["d_down"], None, None)


class MoELayer(torch.nn.Module):
    """Routed SwiGLU experts over the fused layout gate_up [E*H, 2I], down [E*I, H]."""

    def __init__(self, hidden: int, n_experts: int, top_k: int, inter: int, device="cuda"):
        super().__init__()
        self.k = top_k
        self.w_router = torch.nn.Parameter(torch.empty(hidden, n_experts, dtype=torch.float32, device=device))
        self.gate_up = torch.nn.Parameter(torch.empty(n_experts * hidden, 2 * inter, dtype=torch.bfloat16,
                                                      device=device))
        self.down = torch.nn.Parameter(torch.empty(n_experts * inter, hidden, dtype=torch.bfloat16,
                                                   device=device))

    def forward(self, x, bias=None):
        return MoELayerFunction.apply(x, self.w_router, self.gate_up, self.down, self.k, bias)


class ForwardGraph:
    """The layer forward captured once as a CUDA graph, for a fixed token
    count and fixed weights (inference).

    Write a batch's tokens into ``x`` (or pass them to ``__call__``); a replay
    runs route, permute, both grouped GEMMs and the combine as one graph
    launch, with no per-kernel launch gaps, and writes ``y``, which the next
    replay overwrites.  Every step of the path stays on the device (expert
    offsets included), so one capture serves any routing.  The graph keeps
    its intermediates in its own memory pool.

    The weights are fixed for the graph's life: W_r's bf16 split (the tensor
    cores' router operand) is made once here, outside the graph.  After
    changing W_r in place, call ``refresh_router_split()``.
    """

    def __init__(self, T, w_router, gate_up, down, k, bias=None, sh_gate_up=None, sh_down=None,
                 fused_gather=False):
        H, E = w_router.shape
        self.args = (w_router, gate_up, down, k, bias, sh_gate_up, sh_down)
        self.fused_gather = fused_gather
        self.w_split = ops.route_split_weight(w_router) if ops.route_supports_split(H, E) else None
        self.x = torch.zeros((T, H), dtype=torch.bfloat16, device=w_router.device)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):          # one-time library set-up happens outside the capture
            for _ in range(2):
                self._forward()
        torch.cuda.current_stream().wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.y = self._forward()

    def _forward(self):
        w_router, gate_up, down, k, bias, sh_gu, sh_dn = self.args
        y, _ = moe_forward(self.x, w_router, gate_up, down, k, bias, sh_gu, sh_dn,
                           fused_gather=self.fused_gather, w_split=self.w_split)
        return y

    def refresh_router_split(self):
        """Re-derives W_r's split (in place, where the graph reads it) after W_r changed."""
        if self.w_split is not None:
            ops.route_split_weight(self.args[0], out=self.w_split)

    def replay(self):
        """Runs the layer on the current contents of ``x``; returns ``y``."""
        self.graph.replay()
        return self.y

    def __call__(self, x):
        self.x.copy_(x)
        return self.replay()


class PipelinedForward:
    """The forward over a stream of host batches, with copies overlapped.

    Batch i's layer runs on the compute stream while batch i+1's tokens are
    copied host -> device and batch i-1's output device -> host on a copy
    stream (events between the streams).  The layer runs as one of two
    ForwardGraph replays, one per input buffer.  Host tensors must be pinned
    for the copies to be asynchronous; every batch has the token count the
    graphs were captured for.
    """

    def __init__(self, T, w_router, gate_up, down, k, bias=None, sh_gate_up=None, sh_down=None,
                 fused_gather=False):
        self.graphs = [ForwardGraph(T, w_router, gate_up, down, k, bias, sh_gate_up, sh_down,
                                    fused_gather) for _ in range(2)]
        self.copy_stream = torch.cuda.Stream()
        self.ev_loaded = [torch.cuda.Event(), torch.cuda.Event()]
        self.ev_done = [torch.cuda.Event(), torch.cuda.Event()]
        self.ev_stored = [torch.cuda.Event(), torch.cuda.Event()]

    def run(self, x_host_batches, y_host_batches):
        """y_host_batches[i] <- layer(x_host_batches[i]); returns when all are stored."""
        compute = torch.cuda.current_stream()
        n = len(x_host_batches)
        for b in range(2):
            self.ev_done[b].record(compute)     # both buffers free at the start
            self.ev_stored[b].record(compute)

        def load(i):
            b = i % 2
            with torch.cuda.stream(self.copy_stream):
                self.copy_stream.wait_event(self.ev_done[b])     # the layer no longer reads it
                self.graphs[b].x.copy_(x_host_batches[i], non_blocking=True)
                self.ev_loaded[b].record(self.copy_stream)

        if n:
            load(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                load(i + 1)
            compute.wait_event(self.ev_loaded[b])
            compute.wait_event(self.ev_stored[b])                # batch i-2's output was copied out
            y = self.graphs[b].replay()
            self.ev_done[b].record(compute)
            with torch.cuda.stream(self.copy_stream):
                self.copy_stream.wait_event(self.ev_done[b])
                y_host_batches[i].copy_(y, non_blocking=True)
                self.ev_stored[b].record(self.copy_stream)
        self.copy_stream.synchronize()
        compute.synchronize()


class OverlappedForward:
    """The forward over a stream of host batches as a two-stage pipeline, so
    that the token-side steps of one batch overlap the expert GEMMs of the
    previous one (the single-GPU part of the Domino-style overlap: ByteDance
    "FSDPTurbo" domino dispatcher; "InternVL3.5 pure FSDP2 训练性能优化实践").

    Stage F (route -> permute -> row gather) and stage G (grouped gate_up
    GEMM -> grouped down GEMM -> combine, plus the shared expert) are each
    captured as a CUDA graph per buffer set, two sets, and run on their own
    streams: F of batch i+1 runs while G of batch i runs.  Tokens are not
    split within a batch, so every expert's weights are still read once per
    batch.  A copy stream uploads each batch and downloads its output.
    Outputs equal moe_forward's bit for bit.  Host tensors must be pinned;
    every batch has the token count given here.  As ForwardGraph, it makes
    W_r's bf16 split once at construction (``refresh_router_split()`` after
    changing W_r).
    """

    def __init__(self, T, w_router, gate_up, down, k, bias=None, sh_gate_up=None, sh_down=None,
                 fused_gather=False):
        H, E = w_router.shape
        I = down.shape[0] // E
        self.w_router = w_router
        self.w_split = ops.route_split_weight(w_router) if ops.route_supports_split(H, E) else None
        w_split = self.w_split
        self.stream_f = torch.cuda.Stream()
        self.stream_g = torch.cuda.Stream()
        self.copy_stream = torch.cuda.Stream()
        # stage G reads x itself for the shared expert and the fused row gather
        self.g_reads_x = sh_gate_up is not None or fused_gather
        self.sets = []
        for _ in range(2):
            st = {"x": torch.zeros((T, H), dtype=torch.bfloat16, device=w_router.device)}

            def front(st=st):
                ids, w = ops.route(st["x"], w_router, k, bias, w_split=w_split)
                counts, offsets, row_map, src_row = ops.permute(ids, E)
                x_perm = None if fused_gather else ops.permute_rows_scatter(st["x"], row_map, k)
                st.update(w=w, offsets=offsets, row_map=row_map, src_row=src_row, x_perm=x_perm)

            def back(st=st):
                if fused_gather:
                    h, _, _ = ops.grouped_gemm_gate_up_swiglu(st["x"], st["src_row"], st["offsets"], gate_up, I)
                else:
                    h, _, _ = ops.grouped_gemm_gate_up_swiglu(st["x_perm"], None, st["offsets"], gate_up, I)
                y_perm = ops.grouped_gemm_down(h, st["offsets"], down, H)
                y_sh = None
                if sh_gate_up is not None:
                    I_s = sh_down.shape[0]
                    hs, _, _ = ops.grouped_gemm_gate_up_swiglu(st["x"], None, None, sh_gate_up, I_s)
                    y_sh = ops.grouped_gemm_down(hs, None, sh_down, H)
                st["y"] = ops.unpermute_combine(y_perm, st["row_map"], st["w"], y_sh)

            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):      # one-time library set-up outside the captures
                for _ in range(2):
                    front()
                    back()
            torch.cuda.current_stream().wait_stream(side)
            st["gf"], st["gg"] = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            # The two stages run side by side: captured without programmatic
            # dependent launch, whose early-resident kernels would take the
            # SMs that the other stage fills at each GEMM's tail.
            pdl = ops.pdl_enabled()
            ops.set_pdl(False)
            try:
                with torch.cuda.graph(st["gf"]):
                    front()
                with torch.cuda.graph(st["gg"]):
                    back()
            finally:
                ops.set_pdl(pdl)
            st.update(ev_loaded=torch.cuda.Event(), ev_f=torch.cuda.Event(), ev_g=torch.cuda.Event(),
                      ev_stored=torch.cuda.Event())
            self.sets.append(st)

    def refresh_router_split(self):
        """Re-derives W_r's split (in place, where the graphs read it) after W_r changed."""
        if self.w_split is not None:
            ops.route_split_weight(self.w_router, out=self.w_split)

    def run(self, x_host_batches, y_host_batches):
        """y_host_batches[i] <- layer(x_host_batches[i]); returns when all are stored."""
        cur = torch.cuda.current_stream()
        for st in self.sets:                    # every buffer free at the start
            for ev in ("ev_f", "ev_g", "ev_stored"):
                st[ev].record(cur)
        for s in (self.stream_f, self.stream_g, self.copy_stream):
            s.wait_stream(cur)
        n = len(x_host_batches)

        def load(i):
            st = self.sets[i % 2]
            with torch.cuda.stream(self.copy_stream):
                self.copy_stream.wait_event(st["ev_f"])          # F of batch i-2 has read x
                if self.g_reads_x:
                    self.copy_stream.wait_event(st["ev_g"])      # and so has G of batch i-2
                st["x"].copy_(x_host_batches[i], non_blocking=True)
                st["ev_loaded"].record(self.copy_stream)

        if n:
            load(0)
        for i in range(n):
            st = self.sets[i % 2]
            if i + 1 < n:
                load(i + 1)
            with torch.cuda.stream(self.stream_f):
                self.stream_f.wait_event(st["ev_loaded"])
                self.stream_f.wait_event(st["ev_g"])             # G of batch i-2 no longer reads this set
                st["gf"].replay()
                st["ev_f"].record(self.stream_f)
            with torch.cuda.stream(self.stream_g):
                self.stream_g.wait_event(st["ev_f"])
                self.stream_g.wait_event(st["ev_stored"])        # batch i-2's output was copied out
                st["gg"].replay()
                st["ev_g"].record(self.stream_g)
            with torch.cuda.stream(self.copy_stream):
                self.copy_stream.wait_event(st["ev_g"])
                y_host_batches[i].copy_(st["y"], non_blocking=True)
                st["ev_stored"].record(self.copy_stream)
        self.copy_stream.synchronize()
        cur.wait_stream(self.stream_f)
        cur.wait_stream(self.stream_g)
        cur.synchronize()
