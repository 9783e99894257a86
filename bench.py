"""Benchmark of the MoE expert layer on GB300 (one JSON line on rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload qwen3_moe] [--no-fwd-bwd] [--no-cpu-baseline]

A step is one pass of the layer over one batch of synthetic input: route ->
permute -> grouped gate_up GEMM + SwiGLU -> grouped down GEMM -> combine, on
the Qwen3-MoE-shaped workload (T=4096, H=2048, E=128, k=8, I=768) unless
--workload names another.  Inputs and weights are resident in HBM; L2 is
flushed (256 MB write) before every step, outside the timed events.  `value`
is tokens/s over exactly K device-timed steps (CUDA events on the launching
stream), max over ranks; `e2e` repeats the step through the public API with
the tokens copied from pinned host memory and the output copied back inside
the timed region.  A training step (forward + backward) at the training
workload (T=8192) is reported under `fwd_bwd`.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the layer has no data-path exchange on one node here: "replicas only");
ranks meet only at the timing barriers.

--impl reference times the fp64 CPU oracle (the reference arm: a plain, slow
restatement of the layer) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s (fwd; fwd+bwd) and grouped-GEMM % of GB300 bf16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


SPACER_CYCLES = 2_000_000   # about 1 ms of device spin ahead of each eager step


def route_launches(H, E, presplit=False):
    """Kernels of one router call: the bf16 split of W_r (unless made once
    beforehand), then the fused cluster router (16 <= E <= 256, E % 16 == 0)
    or the router GEMM and top-k."""
    return (2 if (H % 64 == 0 and E % 16 == 0 and 16 <= E <= 256) else 3) - (1 if presplit else 0)


def permute_launches(R, torch, device):
    """Kernels of one moe_permute call: one cooperative launch while its
    256-assignment blocks fit on the device at once (8 per SM), else three."""
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    return 1 if (R + 255) // 256 <= 8 * sms else 3


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="qwen3_moe")
    ap.add_argument("--no-fwd-bwd", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-deepseek", action="store_true",
                    help="skip the DeepSeek-V3-shaped forward leg (reported under deepseek_v3)")
    ap.add_argument("--train-only", action="store_true",
                    help="time only the training step (forward + backward) for --steps steps")
    ap.add_argument("--gather", default="rows", choices=["fused", "rows"],
                    help="fused: the gate_up GEMM gathers token rows itself with TMA tile::gather4; "
                         "rows: materialise the permuted rows first and stream them with TMA tiles "
                         "(default, fastest)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------- distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend):
    import torch.distributed as dist

    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if ws > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value, device=None):
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 - 0.05 <= ts <= t1 + 0.05):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        mhz.sort()
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


# ------------------------------------------------------------ native arm

def traffic_for(*kernel_srcs):
    """dram bytes (read + write) per launch of the dominant kernel, from the
    ncu capture summarised in profiles/grouped_gemm_qwen3_moe.md, whose two
    machine-read figures sit beside it in profiles/grouped_gemm_qwen3_moe.json;
    None when the kernel's sources changed since the capture (the JSON holds
    the sha256 of those sources, read in order and concatenated)."""
    path = os.path.join(ROOT, "profiles", "grouped_gemm_qwen3_moe.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        fields = json.load(f)
    h = hashlib.sha256(b"".join(open(f, "rb").read() for f in kernel_srcs)).hexdigest()
    if fields.get("source_sha256") != h or "dram_bytes_per_launch" not in fields:
        return None
    return int(fields["dram_bytes_per_launch"])


def device_inputs(cfg, torch, device):
    import numpy as np

    import synth

    inp = synth.make_inputs(cfg, with_dy=cfg.train)

    def bf(a):
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)

    d = dict(x=bf(inp.x), w_router=torch.from_numpy(inp.w_router).to(device), gate_up=bf(inp.gate_up),
             down=bf(inp.down))
    d["bias"] = torch.from_numpy(inp.bias).to(device) if inp.bias is not None else None
    d["sh_gate_up"] = bf(inp.sh_gate_up) if inp.sh_gate_up is not None else None
    d["sh_down"] = bf(inp.sh_down) if inp.sh_down is not None else None
    d["dy"] = bf(inp.dy) if inp.dy is not None else None
    d["x_host"] = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    return d


def make_step(moe, d, cfg, stream, fused):
    """One forward step of the layer through the public API, with an optional
    list of CUDA events recorded between its kernels (names: what lies
    between consecutive events).  The weights are fixed (inference), so W_r's
    bf16 split for the tensor-core router is made once here, as ForwardGraph
    does, outside every timed region."""
    T, H, E, k, I = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I
    I_s = cfg.I_shared
    w_split = moe.route_split_weight(d["w_router"]) if moe.route_supports_split(H, E) else None
    names = ["route", "permute"] + ([] if fused else ["permute_rows"]) + ["gate_up", "down"] + \
        (["shared"] if I_s else []) + ["combine"]

    def step(ev=None):
        j = [0]

        def mark():
            if ev is not None:
                ev[j[0]].record(stream)
            j[0] += 1
        mark()
        ids, w = moe.route(d["x"], d["w_router"], k, d["bias"], w_split=w_split)
        mark()
        counts, offsets, row_map, src_row = moe.permute(ids, E)
        mark()
        if fused:
            h, _, _ = moe.grouped_gemm_gate_up_swiglu(d["x"], src_row, offsets, d["gate_up"], I)
        else:
            x_perm = moe.permute_rows_scatter(d["x"], row_map, k)
            mark()
            h, _, _ = moe.grouped_gemm_gate_up_swiglu(x_perm, None, offsets, d["gate_up"], I)
        mark()
        y_perm = moe.grouped_gemm_down(h, offsets, d["down"], H)
        mark()
        y_sh = None
        if I_s:
            hs, _, _ = moe.grouped_gemm_gate_up_swiglu(d["x"], None, None, d["sh_gate_up"], I_s)
            y_sh = moe.grouped_gemm_down(hs, None, d["sh_down"], H)
            mark()
        y = moe.unpermute_combine(y_perm, row_map, w, y_sh)
        mark()
        return y

    return names, step


def run_native(args):
    import torch

    import synth
    import token_dispatch_grouped_softmax_gb300 as moe

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist("nccl")
    moe.build()
    moe.load()
    cfg = synth.CONFIGS[args.workload]
    pk, pk_kind = peaks()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    if args.train_only:
        res = fwd_bwd(moe, torch, torch.cuda.current_stream(), dist, device, ws, flush, pk,
                      args.gather != "rows", K=args.steps, W=max(args.warmup, 3))
        if rank == 0:
            print(json.dumps({"metric": METRIC, "fwd_bwd": res}), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    d = device_inputs(cfg, torch, device)
    stream = torch.cuda.current_stream()
    T, H, E, k, I = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I
    I_s = cfg.I_shared

    fused = args.gather == "fused"
    names, step = make_step(moe, d, cfg, stream, fused)

    # route (weight split + fused router, or split + router GEMM + top-k),
    # permute (one cooperative kernel, or three), row gather, gate_up, down,
    # shared expert (2), combine
    launches_per_step = route_launches(H, cfg.E, presplit=True) + permute_launches(T * k, torch, device) + \
        (0 if fused else 1) + 1 + 1 + (2 if I_s else 0) + 1
    for _ in range(max(args.warmup, 3)):
        step()
    moe.sync_status()
    torch.cuda.synchronize()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.time()
    # (1) eager launches with an event between kernels: the per-kernel times.
    # A spin of about a millisecond on the device after the flush lets the
    # host enqueue the whole step before the device reaches it, so the events
    # bracket device time only (no host launch gaps between kernels).
    for i in range(K):
        flush.zero_()
        torch.cuda._sleep(SPACER_CYCLES)
        step(evs[i])
    torch.cuda.synchronize()
    barrier(dist)
    moe.sync_status()
    eager_ms = [evs[i][0].elapsed_time(evs[i][-1]) for i in range(K)]
    per_kernel = {n: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K)) / K
                  for j, n in enumerate(names)}
    eager_s = max_over_ranks(dist, sum(eager_ms) / 1e3, device)
    # (2) the same forward as one CUDA graph per step (ForwardGraph): the value
    graph = moe.ForwardGraph(T, d["w_router"], d["gate_up"], d["down"], k, d["bias"], d["sh_gate_up"],
                             d["sh_down"], fused_gather=fused)
    graph.x.copy_(d["x"])
    for _ in range(max(args.warmup, 3)):
        graph.replay()
    torch.cuda.synchronize()
    barrier(dist)
    gevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush.zero_()
        gevs[i][0].record(stream)
        graph.replay()
        gevs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    t1 = time.time()
    clk = clocks.stop(t0, t1)
    moe.sync_status()
    y_graph_ok = bool(torch.equal(graph.y.view(torch.int16), step().view(torch.int16)))
    del graph
    step_ms = [gevs[i][0].elapsed_time(gevs[i][1]) for i in range(K)]
    total_s = sum(step_ms) / 1e3
    total_s = max_over_ranks(dist, total_s, device)
    value = ws * T * K / total_s
    ms_per_step = 1e3 * total_s / K

    # rooflines.  The forward GEMMs of a routed batch stream every used
    # expert's weights once; at ~256 rows per expert that takes longer at the
    # HBM peak than their FLOPs take at the bf16 peak, so the binding bound is
    # whichever floor is higher.
    ids_c, _w = moe.route(d["x"], d["w_router"], k, d["bias"])
    counts_c = moe.permute(ids_c, E)[0]
    used = int((counts_c > 0).sum().item())
    f_gate_up = 2.0 * cfg.R * H * 2 * I
    f_down = 2.0 * cfg.R * I * H
    b_gate_up = used * H * 2 * I * 2 + cfg.R * H * 2 + cfg.R * I * 2   # weights + A rows + h
    gemm_ms = per_kernel["gate_up"] + per_kernel["down"] + per_kernel.get("shared", 0.0)
    gemm_flops = cfg.flops_fwd()
    peak_tf = pk["bf16_tflops"]
    dur_s = per_kernel["gate_up"] * 1e-3
    t_hbm, t_tc = b_gate_up / (pk["hbm_gbs"] * 1e9), f_gate_up / (peak_tf * 1e12)
    csrc = os.path.join(ROOT, "token_dispatch_grouped_softmax_gb300", "csrc")
    srcs = [os.path.join(csrc, "grouped_gemm.cu"), os.path.join(csrc, "common.cuh")]
    tensor_part = {"achieved": round(f_gate_up / dur_s / 1e12, 1), "peak": peak_tf, "unit": "TFLOP/s",
                   "frac": round(f_gate_up / dur_s / 1e12 / peak_tf, 4),
                   "algorithmic_flops_per_launch": f_gate_up,
                   "peak_kind": "%s burst bf16 (MEASURED_PEAKS.json)" % pk_kind}
    hbm_part = {"achieved": round(b_gate_up / dur_s / 1e9, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(b_gate_up / dur_s / 1e9 / pk["hbm_gbs"], 4),
                "algorithmic_bytes_per_launch": b_gate_up,
                "peak_kind": "%s HBM copy (MEASURED_PEAKS.json)" % pk_kind}
    main, other = (hbm_part, tensor_part) if t_hbm >= t_tc else (tensor_part, hbm_part)
    roofline = dict({"bound": "hbm" if t_hbm >= t_tc else "tensor",
                     "kernel": "grouped_gemm_kernel<FWD_GATEUP>"}, **main)
    roofline["traffic"] = traffic_for(*srcs)
    roofline["floors_us"] = {"hbm": round(t_hbm * 1e6, 1), "tensor": round(t_tc * 1e6, 1)}
    roofline["other_bound"] = dict({"bound": "tensor" if t_hbm >= t_tc else "hbm"}, **other)
    roofline["experts_used"] = used
    comb_bytes = cfg.R * H * 2 + T * H * 2 + cfg.R * 8
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "T": T, "H": H, "E": E, "k": k, "I": I, "I_shared": I_s,
                   "seed": cfg.seed, "description": cfg.description,
                   "l2": "flushed before every step (256 MB write), outside the timed events",
                   "parallelism": "replicas" if ws > 1 else "single",
                   "gather": args.gather},
        "roofline": roofline,
        "timing": "value and ms_per_step: the forward replayed as one CUDA graph per step "
                  "(ForwardGraph), CUDA events around each replay; kernels_us and eager: the same "
                  "kernels launched one by one with an event between kernels, enqueued behind a "
                  "device-side spin so that no host launch gap falls between the events",
        "eager": {"value": round(ws * T * K / eager_s, 1), "ms_per_step": round(1e3 * eager_s / K, 4)},
        "graph_output_matches_eager": y_graph_ok,
        "kernels_us": {n: round(v * 1e3, 2) for n, v in per_kernel.items()},
        "gemm": {"tflops": round(gemm_flops / (gemm_ms * 1e-3) / 1e12, 1),
                 "frac_of_peak": round(gemm_flops / (gemm_ms * 1e-3) / 1e12 / peak_tf, 4),
                 "down_tflops": round(f_down / (per_kernel["down"] * 1e-3) / 1e12, 1)},
        "combine": {"gbs": round(comb_bytes / (per_kernel["combine"] * 1e-3) / 1e9, 1),
                    "frac_of_hbm": round(comb_bytes / (per_kernel["combine"] * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                    "algorithmic_bytes": comb_bytes},
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "wall_s": round(t1 - t0, 3),
    }

    if not args.no_e2e:
        e_pipe = e2e(moe, d, cfg, torch, stream, dist, device, ws, min(K, 100), fused, "PipelinedForward")
        e_over = e2e(moe, d, cfg, torch, stream, dist, device, ws, min(K, 100), fused, "OverlappedForward")
        out["e2e"] = e_over
        out["e2e_pipelined"] = {k_: e_pipe[k_] for k_ in ("value", "api")}
    if not args.no_fwd_bwd:
        del d
        torch.cuda.empty_cache()
        out["fwd_bwd"] = fwd_bwd(moe, torch, stream, dist, device, ws, flush, pk, fused)
    if not args.no_deepseek and args.workload != "deepseek_v3":
        torch.cuda.empty_cache()
        out["deepseek_v3"] = large_forward(moe, torch, stream, dist, device, ws, flush, pk, fused,
                                           "deepseek_v3")
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg, target_s=15.0)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def e2e(moe, d, cfg, torch, stream, dist, device, ws, K, fused, runner_cls="OverlappedForward"):
    """Tokens from pinned host memory -> layer -> output back to pinned host memory,
    through a public pipelined forward (PipelinedForward: copies of neighbouring
    steps overlap the layer; OverlappedForward: also the route/permute of step
    i+1 overlaps the expert GEMMs of step i).  Every step's input upload and
    output download is inside the timed region."""
    T, H = cfg.T, cfg.H
    runner = getattr(moe, runner_cls)(T, d["w_router"], d["gate_up"], d["down"], cfg.k, d["bias"],
                                      d["sh_gate_up"], d["sh_down"], fused_gather=fused)
    xs = [d["x_host"]] * K
    ys = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    ys = [ys[i % 2] for i in range(K)]
    runner.run(xs[:3], ys[:3])
    torch.cuda.synchronize()
    barrier(dist)
    t0 = time.perf_counter()
    runner.run(xs, ys)
    dt = time.perf_counter() - t0
    barrier(dist)
    s = max_over_ranks(dist, dt, device)
    del runner
    return {"value": round(ws * T * K / s, 1), "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2,
            "d2h_bytes_per_step": T * H * 2, "steps": K, "api": runner_cls,
            "note": "weights resident; every step copies x host->device (pinned) and y device->host "
                    "(pinned); host wall clock around K steps with all streams synchronised"}


def fwd_bwd(moe, torch, stream, dist, device, ws, flush, pk, fused, K=30, W=3):
    """Training step (forward with saved activations + backward) on the training workload."""
    import synth

    cfg = synth.CONFIGS["qwen3_moe_train"]
    d = device_inputs(cfg, torch, device)

    def step():
        y, st = moe.moe_forward(d["x"], d["w_router"], d["gate_up"], d["down"], cfg.k, save_for_backward=True,
                                fused_gather=fused)
        g = moe.moe_backward(d["dy"], st, d["w_router"], d["gate_up"], d["down"])
        return g

    for _ in range(W):
        step()
    moe.sync_status()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(dist)
    for i in range(K):
        flush.zero_()
        torch.cuda._sleep(SPACER_CYCLES)   # the host enqueues ahead of the device (see the forward)
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    moe.sync_status()
    s = sum(a.elapsed_time(b) for a, b in evs) / 1e3
    s = max_over_ranks(dist, s, device)
    flops = 3.0 * cfg.flops_fwd()
    return {"workload": cfg.name, "T": cfg.T, "value": round(ws * cfg.T * K / s, 1), "unit": "tokens/s",
            "ms_per_step": round(1e3 * s / K, 4), "gemm_flops_per_step": flops,
            "layer_tflops": round(flops * K / s / 1e12, 1), "steps": K,
            "launches_per_step": route_launches(cfg.H, cfg.E) + permute_launches(cfg.T * cfg.k, torch, device) + 3 +
                                 (0 if fused else 1) + 1 + 1 + 2 + 2 + 2}


def large_forward(moe, torch, stream, dist, device, ws, flush, pk, fused, name, K=10, K_eager=3, W=3):
    """The forward of a second, larger workload (the DeepSeek-V3 shape: 256
    experts, I = 2048, a shared expert; ~512 rows per expert, so its GEMMs are
    bound by the tensor cores): K graph-replayed steps for tokens/s, and
    K_eager eager steps with an event between kernels for each GEMM's
    TFLOP/s and the combine's GB/s.  L2 flushed before every step."""
    import synth

    cfg = synth.CONFIGS[name]
    d = device_inputs(cfg, torch, device)
    names, step = make_step(moe, d, cfg, stream, fused)
    for _ in range(W):
        step()
    moe.sync_status()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(K_eager)]
    barrier(dist)
    for i in range(K_eager):
        flush.zero_()
        torch.cuda._sleep(SPACER_CYCLES)
        step(evs[i])
    torch.cuda.synchronize()
    per = {n: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K_eager)) / K_eager
           for j, n in enumerate(names)}
    graph = moe.ForwardGraph(cfg.T, d["w_router"], d["gate_up"], d["down"], cfg.k, d["bias"], d["sh_gate_up"],
                             d["sh_down"], fused_gather=fused)
    graph.x.copy_(d["x"])
    for _ in range(W):
        graph.replay()
    torch.cuda.synchronize()
    barrier(dist)
    gevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush.zero_()
        gevs[i][0].record(stream)
        graph.replay()
        gevs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    moe.sync_status()
    s = max_over_ranks(dist, sum(a.elapsed_time(b) for a, b in gevs) / 1e3, device)
    del graph
    T, H, I, R, I_s = cfg.T, cfg.H, cfg.I, cfg.R, cfg.I_shared
    peak = pk["bf16_tflops"]
    flops = {"gate_up": 2.0 * R * H * 2 * I, "down": 2.0 * R * I * H,
             "shared": 2.0 * T * H * 2 * I_s + 2.0 * T * I_s * H}

    def tf(n):
        return round(flops[n] / (per[n] * 1e-3) / 1e12, 1)
    gemm_ms = sum(per[n] for n in flops if n in per)
    comb_bytes = R * H * 2 + T * H * 2 + R * 8 + (T * H * 2 if I_s else 0)
    del d
    torch.cuda.empty_cache()
    return {"workload": cfg.name, "T": T, "H": H, "E": cfg.E, "k": cfg.k, "I": I, "I_shared": I_s,
            "value": round(ws * T * K / s, 1), "unit": "tokens/s", "ms_per_step": round(1e3 * s / K, 4),
            "steps": K, "timing": "value: one CUDA graph replay per step; kernels: eager launches with "
                                  "events between kernels, %d steps" % K_eager,
            "kernels_us": {n: round(v * 1e3, 2) for n, v in per.items()},
            "gemm": {n: {"tflops": tf(n), "frac_of_peak": round(tf(n) / peak, 4)} for n in flops if n in per},
            "gemm_all": {"tflops": round(sum(flops.values()) / (gemm_ms * 1e-3) / 1e12, 1),
                         "frac_of_peak": round(sum(flops.values()) / (gemm_ms * 1e-3) / 1e12 / peak, 4)},
            "combine": {"gbs": round(comb_bytes / (per["combine"] * 1e-3) / 1e9, 1),
                        "frac_of_hbm": round(comb_bytes / (per["combine"] * 1e-3) / 1e9 / pk["hbm_gbs"], 4)},
            "peak_tflops": peak,
            "gpu_launches": K * (route_launches(H, cfg.E, presplit=True) + permute_launches(R, torch, device) +
                                 (0 if fused else 1) + 2 + (2 if I_s else 0) + 1)}


# -------------------------------------------------------------- CPU oracle

def cpu_baseline(cfg, target_s=15.0, max_tokens=None):
    """The fp64 oracle as it stands, on a bounded token sample of the workload:
    route + per-token expert FFNs + combine for n tokens; tokens/s."""
    import numpy as np

    import oracle
    import synth

    inp = synth.make_inputs(cfg)
    cores = oracle.threads()   # OpenMP threads of the oracle's loops

    def run(n):
        x = np.ascontiguousarray(inp.x[:n])
        t = time.perf_counter()
        r = oracle.route(x, inp.w_router, inp.bias, cfg.k)
        oracle.forward_tokens(np.arange(n), x, inp.gate_up, inp.down, r["ids"], r["w"], inp.sh_gate_up,
                              inp.sh_down)
        return time.perf_counter() - t

    n0 = 32
    t_pilot = run(n0)
    n = int(min(cfg.T if max_tokens is None else max_tokens, max(n0, n0 * target_s / max(t_pilot, 1e-6))))
    dt = run(n) if n != n0 else t_pilot
    return {"value": round(n / dt, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "first %d of %d tokens of %s (route + per-token expert FFNs + combine, fp64), %.1f s"
                      % (n, cfg.T, cfg.name, dt)}


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import synth

    cfg = synth.CONFIGS[args.workload]
    K, W = args.steps, max(args.warmup, 0)
    # bounded: each step a sample sized so that the whole run takes a few
    # minutes (at least 0.5 s a step: enough tokens per core that the
    # oracle's per-token rate holds; smaller samples leave cores idle)
    per_step_s = max(0.5, 120.0 / max(K + W, 1))
    base = cpu_baseline(cfg, target_s=per_step_s)
    n = int(base["sample"].split()[1])
    import numpy as np

    import oracle

    inp = synth.make_inputs(cfg)
    x = np.ascontiguousarray(inp.x[:n])

    def step():
        r = oracle.route(x, inp.w_router, inp.bias, cfg.k)
        oracle.forward_tokens(np.arange(n), x, inp.gate_up, inp.down, r["ids"], r["w"], inp.sh_gate_up,
                              inp.sh_down)

    for _ in range(W):
        step()
    t = time.perf_counter()
    for _ in range(K):
        step()
    dt = time.perf_counter() - t
    value = n * K / dt
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws,
           "steps": K, "warmup": W, "ms_per_step": round(1e3 * dt / K, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k, "I": cfg.I,
                      "I_shared": cfg.I_shared, "seed": cfg.seed},
           "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": oracle.threads(),
                            "kind": "oracle",
                            "sample": "first %d of %d tokens per step (fp64 oracle, route + experts + combine)"
                                      % (n, cfg.T)},
           "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
