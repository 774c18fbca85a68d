"""Benchmark of the Q4_K dequant-fused matmul on one or more GPUs.

Headline: the decode sweep -- M = 1 GEMV over the seven Qwen3-4B layer shapes
(q, k, v, o, gate, up, down) of all 36 layers, 2.04 GB of distinct seeded Q4_K
weights resident in HBM (larger than L2, so every call streams from HBM), one
CUDA-graph replay per step.  The calls follow a decoder layer's data flow:
q, k and v read one activation vector and run as one batched launch, o reads
its own, gate and up read one (one batched launch), down its own -- four
dependent launches per layer.  value = weight bytes streamed / time (GB/s).
The same weights through seven single-matrix launches per layer are reported
beside it ("decode_7call").
Second object: the long-prompt prefill sweep at M = 2048 over the same
weights (tcgen05 path), TFLOP/s = 2*M*N*K / time, in the same four launches
per layer (q/k/v and gate/up as batched GEMMs); the seven-call sweep beside
it ("prefill_7call").

Multi-GPU: replicas only.  Each rank runs the same sweep on its own GPU with
no collective on the data path; value = bytes all ranks streamed / max time.

--impl reference times the CPU oracle (single thread, fp64) on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

SHAPES = synthetic.LAYER_SHAPES
N_LAYERS = synthetic.N_LAYERS
M_PREFILL = 2048


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=N_LAYERS)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--per-shape", action="store_true", help="also time each shape alone")
    ap.add_argument("--crossover", action="store_true",
                    help="also time the GEMV (M = 1) and the tcgen05 GEMM at small M on two layer shapes")
    ap.add_argument("--tc-rates", action="store_true",
                    help="only measure tensor-core instruction rates (tcgen05 kind::f16, mma.sync f16 and s8)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def weight_bytes(N, K):
    return N * (K // 256) * 144


# ------------------------------------------------------------ clock sampler --
class ClockSampler:
    """nvidia-smi streaming SM clocks and throttle reasons every 20 ms; `mark()` brackets
    the timed region, and only the samples read inside it are summarised."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, interval_ms=20):
        self.index = index
        self.interval_ms = interval_ms
        self.rows = []  # (host time, fields)
        self.window = [None, None]
        self._p = None
        self._t = None

    def _read(self):
        for line in self._p.stdout:
            f = [c.strip() for c in line.strip().split(",")]
            if len(f) >= 9:
                self.rows.append((time.perf_counter(), f))

    def __enter__(self):
        try:
            self._p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                        "--format=csv,noheader,nounits", f"-lms={self.interval_ms}"],
                                       stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)  # first samples before the timed region
        except Exception:
            self._p = None
        return self

    def mark(self, start):
        self.window[0 if start else 1] = time.perf_counter()

    def __exit__(self, *a):
        time.sleep(2 * self.interval_ms / 1000)
        if self._p is not None:
            self._p.terminate()
            try:
                self._p.wait(timeout=5)
            except Exception:
                self._p.kill()
            self._t.join(timeout=5)

    def summary(self):
        t0, t1 = self.window
        rows = [f for t, f in self.rows if t0 is not None and t1 is not None and t0 <= t <= t1 + 0.03]
        where = "timed region"
        if not rows and self.rows:
            rows = [min(self.rows, key=lambda r: abs(r[0] - (t0 or 0)))[1]]
            where = "nearest sample to the timed region"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if len(r) > 5 + i and r[5 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "window": where}


# ---------------------------------------------------------------- our arm --
# Groups of matrices that read one activation vector in a decoder layer.
GROUPS = (("qkv", (0, 1, 2)), ("o", (3,)), ("ffn", (4, 5)), ("down", (6,)))


def profiled_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary in profiles/, or None
    when the kernel's sources no longer hash to the value recorded with the counters."""
    import glob
    import hashlib
    import re

    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for m in re.finditer(r"<!-- traffic kernel=(\S+) sources=(\S+) sha256_16=(\S+) bytes_per_launch=(\d+) -->",
                             open(path).read()):
            if m.group(1) != kernel:
                continue
            h = hashlib.sha256()
            try:
                for f in m.group(2).split(","):
                    h.update(open(os.path.join(ROOT, "bit_q4_weight_gb300", "csrc", f), "rb").read())
            except OSError:
                return None
            return int(m.group(4)) if h.hexdigest()[:16] == m.group(3) else None
    return None


def group_index(idx):
    """Index in GROUPS of the group that shape `idx` belongs to."""
    return next(gi for gi, (_, members) in enumerate(GROUPS) if idx in members)


def build_inputs(torch, dev, layers):
    """Seeded weights (host numpy -> device), one activation per layer and group, outputs."""
    W, Y, meta = [], [], []
    XG = []  # per layer: {group: x}
    for layer in range(layers):
        for idx, (name, K, N) in enumerate(SHAPES):
            w = synthetic.q4k_weights(N, K, synthetic.weight_seed(1, layer, idx))
            W.append(torch.from_numpy(w).to(dev))
            Y.append(torch.empty(N, dtype=torch.float32, device=dev))
            meta.append((name, K, N))
        xg = {}
        for gi, (gname, members) in enumerate(GROUPS):
            K = SHAPES[members[0]][1]
            xg[gname] = torch.from_numpy(
                synthetic.activations(1, K, synthetic.activation_seed(1, layer * 8 + gi)).reshape(K)).to(dev)
        XG.append(xg)
    return W, XG, Y, meta


def decode_plan(W, XG, Y, meta, batched):
    """The calls of one decode step: (weights, x, outputs, Ns, K) per launch."""
    plan = []
    for layer, xg in enumerate(XG):
        base = layer * len(SHAPES)
        for gname, members in GROUPS:
            idx = [base + m for m in members]
            K = meta[idx[0]][1]
            calls = [idx] if batched else [[i] for i in idx]
            for c in calls:
                plan.append(([W[i] for i in c], xg[gname], [Y[i] for i in c], [meta[i][2] for i in c], K))
    return plan


def run_plan(q, plan):
    for ws, x, ys, ns, K in plan:
        if len(ws) == 1:
            q.jllm_q4k_gemv(ws[0], x, ns[0], K, out=ys[0])
        else:
            q.jllm_q4k_gemv_batch(ws, x, ns, K, outs=ys)


def max_over_ranks(torch, dist, t, world, device=None):
    """Seconds maxed over the ranks: the slowest replica sets the job's time (a collective
    over the timing only; the data path has none)."""
    if world <= 1:
        return t
    tt = torch.tensor([float(t)], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def time_graph(torch, graph, stream, steps, warmup, clk=None):
    """Seconds per replay, CUDA events recorded on the stream the graph is launched on."""
    with torch.cuda.stream(stream):
        for _ in range(warmup - 1):
            graph.replay()
        torch.cuda.synchronize()
        # the last warm-up replay stays in flight, so that the timed replays are queued
        # behind it and the start event does not time the host's first submission
        graph.replay()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        if clk:
            clk.mark(True)
        start.record(stream)
        for _ in range(steps):
            graph.replay()
        end.record(stream)
    end.synchronize()
    if clk:
        clk.mark(False)
    return start.elapsed_time(end) / 1e3 / steps


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__

    __graft_entry__.build()
    import bit_q4_weight_gb300 as q

    layers = args.layers
    W, XG, Y, meta = build_inputs(torch, dev, layers)
    total_bytes = sum(weight_bytes(N, K) for (_, K, N) in meta)
    plan = decode_plan(W, XG, Y, meta, batched=True)
    n_launch = len(plan)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def capture(p):
        with torch.cuda.stream(stream):
            run_plan(q, p)  # eager warm-up (first launches set kernel attributes)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run_plan(q, p)
        torch.cuda.synchronize()
        return g

    def sync_ranks():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    def tmax(t):
        return max_over_ranks(torch, dist, t, world, dev)

    g = capture(plan)
    sync_ranks()
    with ClockSampler(local) as clk:
        t_step = time_graph(torch, g, stream, args.steps, args.warmup, clk)
    clocks = clk.summary()
    sync_ranks()
    t_max = tmax(t_step)
    value = total_bytes * world / t_max / 1e9
    del g

    # the same sweep as ONE call: jllm_q4k_gemv_chain (one persistent launch for the 144 steps)
    chain = q.GemvChain(plan)
    with torch.cuda.stream(stream):
        chain(stream)
    torch.cuda.synchronize()
    gc = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gc, stream=stream):
        chain(stream)
    torch.cuda.synchronize()
    sync_ranks()
    tc = tmax(time_graph(torch, gc, stream, args.steps, args.warmup))
    del gc

    # the same weights, seven single-matrix launches per layer
    plan7 = decode_plan(W, XG, Y, meta, batched=False)
    g7 = capture(plan7)
    sync_ranks()
    t7 = tmax(time_graph(torch, g7, stream, args.steps, args.warmup))
    del g7

    # the same batched sweep with the RMSNorm prologue on the q/k/v and gate/up launches
    # (their x is then the un-normalised residual stream; one fp32 gamma per group and layer)
    gammas = [{gname: torch.from_numpy(np.random.Generator(np.random.PCG64(7000 + 4 * l + gi))
                                       .uniform(0.25, 2.0, size=meta[l * len(SHAPES) + members[0]][1])
                                       .astype(np.float32)).to(dev)
               for gi, (gname, members) in enumerate(GROUPS) if len(members) > 1} for l in range(layers)]
    plan_n = []
    for (ws, x, ys, ns, K), (layer, gname) in zip(plan, [(l, gn) for l in range(layers) for gn, _ in GROUPS]):
        plan_n.append((ws, x, ys, ns, K, gammas[layer].get(gname)))

    def run_plan_norm():
        for ws, x, ys, ns, K, gm in plan_n:
            if gm is not None:
                q.jllm_q4k_gemv_rmsnorm_batch(ws, x, gm, 1e-6, ns, K, outs=ys)
            elif len(ws) == 1:
                q.jllm_q4k_gemv(ws[0], x, ns[0], K, out=ys[0])
            else:
                q.jllm_q4k_gemv_batch(ws, x, ns, K, outs=ys)

    with torch.cuda.stream(stream):
        run_plan_norm()
    torch.cuda.synchronize()
    gn = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gn, stream=stream):
        run_plan_norm()
    torch.cuda.synchronize()
    sync_ranks()
    tn = tmax(time_graph(torch, gn, stream, args.steps, args.warmup))
    del gn

    # the same sweep with the attention input block of Qwen3 fused into the q/k/v launch:
    # RMSNorm of x, the three projections, per-head RMSNorm of q and k, RoPE at a position
    hg = [torch.from_numpy(np.random.Generator(np.random.PCG64(7500 + l)).uniform(0.5, 1.5, size=(2, 128))
                           .astype(np.float32)).to(dev) for l in range(layers)]
    n_q_heads, n_kv_heads = SHAPES[0][2] // 128, SHAPES[1][2] // 128

    def run_plan_rope():
        for (ws, x, ys, ns, K, gm), (layer, gname) in zip(plan_n, [(l, gn) for l in range(layers) for gn, _ in GROUPS]):
            if gname == "qkv":
                q.jllm_q4k_gemv_qkv_rope(ws, x, n_q_heads, n_kv_heads, K, 1000 + layer, 1e6, gamma=gm, eps=1e-6,
                                         q_gamma=hg[layer][0], k_gamma=hg[layer][1], head_eps=1e-6, outs=ys)
            elif gm is not None:
                q.jllm_q4k_gemv_rmsnorm_batch(ws, x, gm, 1e-6, ns, K, outs=ys)
            elif len(ws) == 1:
                q.jllm_q4k_gemv(ws[0], x, ns[0], K, out=ys[0])
            else:
                q.jllm_q4k_gemv_batch(ws, x, ns, K, outs=ys)

    with torch.cuda.stream(stream):
        run_plan_rope()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        run_plan_rope()
    torch.cuda.synchronize()
    sync_ranks()
    tr = tmax(time_graph(torch, gr, stream, args.steps, args.warmup))
    del gr

    # end to end: host->device copy of every activation, the sweep, device->host of every output
    xs_flat = [xg[gname] for xg in XG for gname, _ in GROUPS]
    xs_host = torch.cat([x.cpu() for x in xs_flat]).pin_memory()
    ys_host = torch.empty(sum(y.numel() for y in Y), dtype=torch.float32).pin_memory()
    x_dev_all = torch.empty_like(xs_host, device=dev)
    y_dev_all = torch.empty(ys_host.numel(), dtype=torch.float32, device=dev)
    offs_x = np.cumsum([0] + [x.numel() for x in xs_flat])
    offs_y = np.cumsum([0] + [y.numel() for y in Y])
    XGv = [{gname: x_dev_all[offs_x[l * len(GROUPS) + gi]:offs_x[l * len(GROUPS) + gi + 1]]
            for gi, (gname, _) in enumerate(GROUPS)} for l in range(layers)]
    Yv = [y_dev_all[offs_y[i]:offs_y[i + 1]] for i in range(len(Y))]
    ge = capture(decode_plan(W, XGv, Yv, meta, batched=True))

    def e2e_step():
        with torch.cuda.stream(stream):
            x_dev_all.copy_(xs_host, non_blocking=True)
            ge.replay()
            ys_host.copy_(y_dev_all, non_blocking=True)
        stream.synchronize()

    for _ in range(args.warmup):
        e2e_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    t_e2e = tmax((time.perf_counter() - t0) / args.steps)
    e2e = {"value": round(total_bytes * world / t_e2e / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": int(xs_host.numel() * 2), "d2h_bytes_per_step": int(ys_host.numel() * 4),
           "how": "per step: pinned host -> device copy of the step's activations, a CUDA-graph replay of "
                  "the 144 C-ABI calls, device -> host copy of every output, stream synchronize"}
    del ge

    # the same end to end with every C-ABI call made eagerly from the host each step (no graph):
    # ctypes marshalling, the library's argument checks and launches are all inside the step
    plan_e = decode_plan(W, XGv, Yv, meta, batched=True)

    def e2e_eager_step():
        with torch.cuda.stream(stream):
            x_dev_all.copy_(xs_host, non_blocking=True)
            run_plan(q, plan_e)
            ys_host.copy_(y_dev_all, non_blocking=True)
        stream.synchronize()

    for _ in range(args.warmup):
        e2e_eager_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_eager_step()
    t_eager = tmax((time.perf_counter() - t0) / args.steps)
    e2e["eager"] = {"value": round(total_bytes * world / t_eager / 1e9, 2), "unit": "GB/s",
                    "ms_per_step": round(t_eager * 1e3, 4),
                    "how": "the same copies, the 144 C-ABI calls issued eagerly from Python (ctypes) every step"}

    # the same end to end through ONE eager C-ABI call per step: jllm_q4k_gemv_chain
    chain_e = q.GemvChain(decode_plan(W, XGv, Yv, meta, batched=True))

    def e2e_chain_step():
        with torch.cuda.stream(stream):
            x_dev_all.copy_(xs_host, non_blocking=True)
            chain_e(stream)
            ys_host.copy_(y_dev_all, non_blocking=True)
        stream.synchronize()

    for _ in range(args.warmup):
        e2e_chain_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_chain_step()
    t_ce = tmax((time.perf_counter() - t0) / args.steps)
    e2e["chain_eager"] = {"value": round(total_bytes * world / t_ce / 1e9, 2), "unit": "GB/s",
                          "ms_per_step": round(t_ce * 1e3, 4),
                          "how": "the same copies around one eager jllm_q4k_gemv_chain call (all 144 steps)"}

    peaks = {}
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk_path):
        peaks = json.load(open(pk_path))
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    peak_note = "measured" if "hbm_gbs" in peaks else "fallback"

    per_shape = {}
    if args.per_shape and rank == 0:
        for idx, (name, K, N) in enumerate(SHAPES):
            sel = [i for i in range(len(W)) if i % len(SHAPES) == idx]
            gname = next(gn for gn, members in GROUPS if idx in members)
            gs = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gs, stream=stream):
                for i in sel:
                    q.jllm_q4k_gemv(W[i], XG[i // len(SHAPES)][gname], N, K, out=Y[i])
            torch.cuda.synchronize()
            t = time_graph(torch, gs, stream, max(3, args.steps // 2), 3)
            per_shape[name] = round(len(sel) * weight_bytes(N, K) / t / 1e9, 1)
            del gs

    crossover = None
    if args.crossover and rank == 0:
        crossover = run_crossover(torch, q, W, meta, dev, stream, args)

    prefill = None
    ffn = None
    short = None
    kv = run_kv_codec(torch, q, dev, stream, args) if rank == 0 else None
    if not args.no_prefill:
        prefill = run_prefill(torch, q, W, meta, dev, stream, args, world, tmax=tmax, sync=sync_ranks)
        if rank == 0:
            ffn = run_ffn_lmhead(torch, q, W, dev, stream, args)
            # 33 and 235 are the short-prompt workload's sizes; 8 and 16 show the few-token GEMM
            short = {f"M{m}": run_prefill(torch, q, W, meta, dev, stream, args, world, M=m, short=True)
                     for m in (8, 16, 33, 235)}
            prefill["other_M"] = {f"M{m}": run_prefill(torch, q, W, meta, dev, stream, args, world, M=m, light=True)
                                  for m in (1024, 3072)}
            short["workload"] = ("short-prompt prefill over the decode sweep's weights, per-token scaled X, "
                                 "fp16 out, 4 launches per layer (qkv and gate/up batched); M = 33 and 235 the "
                                 "short-prompt sizes, M = 8 and 16 beside them")

    if rank == 0:
        line = {
            "metric": "Q4_K matmul: M=1 weight GB/s vs HBM peak; M=2048 TFLOP/s vs BF16 peak",
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(t_max * 1e3, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "q4k-f16-f32",
            "data": "synthetic (seeded GGUF Q4_K blocks, fp16 N(0,1) activations)",
            "config": {"workload": f"decode sweep M=1, {layers} layers x 7 Qwen3-4B shapes "
                                   "(q/k/v and gate/up batched on their shared x: 4 launches per layer)",
                       "weight_bytes_per_step": total_bytes, "launches_per_step": n_launch,
                       "l2": f"inputs larger than L2 ({total_bytes / 1e9:.2f} GB of weights cycled)", "parallelism": f"replicas{world}"},
            "gpu_launches": n_launch * args.steps,
            "clocks": clocks,
            "roofline": {"bound": "hbm", "achieved": round(total_bytes / t_step / 1e9, 2), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(total_bytes / t_step / 1e9 / hbm_peak, 4),
                         "traffic": profiled_traffic("q4k_gemv_kernel"), "peak_source": peak_note,
                         "bytes_per_launch": round(total_bytes / n_launch),
                         "kernel": "q4k_gemv_kernel", "avg_launch_us": round(t_step / n_launch * 1e6, 3),
                         "frac_of_nominal_7900": round(total_bytes / t_step / 1e9 / 7900.0, 4)},
            "e2e": e2e,
            "decode_chain": {"value": round(total_bytes * world / tc / 1e9, 2), "unit": "GB/s",
                             "ms_per_step": round(tc * 1e3, 4), "launches_per_step": 1,
                             "workload": "the batched decode sweep (144 steps) as one jllm_q4k_gemv_chain call"},
            "decode_7call": {"value": round(total_bytes * world / t7 / 1e9, 2), "unit": "GB/s",
                             "ms_per_step": round(t7 * 1e3, 4), "launches_per_step": len(plan7)},
            "decode_rmsnorm_fused": {"value": round(total_bytes * world / tn / 1e9, 2), "unit": "GB/s",
                                     "ms_per_step": round(tn * 1e3, 4), "launches_per_step": len(plan_n),
                                     "workload": "the batched decode sweep with RMSNorm(x) in the prologue of "
                                                 "the q/k/v and gate/up launches"},
            "decode_qkv_rope_fused": {"value": round(total_bytes * world / tr / 1e9, 2), "unit": "GB/s",
                                      "ms_per_step": round(tr * 1e3, 4), "launches_per_step": len(plan_n),
                                      "workload": "decode_rmsnorm_fused with the q/k/v launch also applying "
                                                  "Qwen3's per-head RMSNorm of q and k and RoPE (base 1e6) "
                                                  "in its epilogue (jllm_q4k_gemv_qkv_rope)"},
        }
        if per_shape:
            line["per_shape_gbs"] = per_shape
        if crossover:
            line["crossover"] = crossover
        if prefill:
            line["prefill_m2048"] = prefill
            if short:
                line["prefill_short"] = short
        if ffn:
            line["ffn_lmhead"] = ffn
        if kv:
            line["kv_codec"] = kv
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(budget_s=12.0)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_crossover(torch, q, W, meta, dev, stream, args):
    """Weight GB/s and TFLOP/s of jllm_q4k_gemm as M grows (fp16 out, workspace when one is
    used), for the q (2560->4096) and gate (2560->9728) shapes over all layers, and the
    M = 1 GEMV -- the evidence for the dispatch threshold (run once per threshold with
    JLLM_GEMV_MAX_M to compare the two paths at the same M)."""
    out = {}
    for shape_idx in (0, 4):
        name, K, N = SHAPES[shape_idx]
        sel = [i for i in range(len(W)) if i % len(SHAPES) == shape_idx]
        wbytes = len(sel) * weight_bytes(N, K)
        res = {}
        for M in (1, 2, 4, 8, 16, 33, 64, 128, 235):
            x = torch.from_numpy(synthetic.activations(M, K, synthetic.activation_seed(2, M, shape_idx))).to(dev)
            paths = [("gemv", None)] if M == 1 else [("gemm", q.workspace(M, N, K, dev))]
            for path, ws in paths:
                if path == "gemv":
                    y = torch.empty(N, dtype=torch.float32, device=dev)
                    call = lambda w: q.jllm_q4k_gemv(w, x.view(K), N, K, out=y)
                else:
                    y = torch.empty((M, N), dtype=torch.float16, device=dev)
                    wsp, wsn = (ws.data_ptr(), ws.numel()) if ws is not None else (None, 0)
                    call = lambda w: q.lib.jllm_q4k_gemm(w.data_ptr(), x.data_ptr(), y.data_ptr(), 1, M, N, K,
                                                         wsp, wsn, stream.cuda_stream)
                with torch.cuda.stream(stream):
                    for i in sel:
                        call(W[i])
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in sel:
                        call(W[i])
                torch.cuda.synchronize()
                t = time_graph(torch, g, stream, 10, 3)
                del g
                res[f"{path}_M{M}"] = {"weight_gbs": round(wbytes / t / 1e9, 1),
                                       "tflops": round(2.0 * M * N * K * len(sel) / t / 1e12, 2)}
        out[f"{name}_{K}x{N}"] = res
    return out


def run_kv_codec(torch, q, dev, stream, args):
    """FP16 <-> INT8 KV codec over a 4096-token Qwen3-4B cache: 36 layers x {K, V} x 8 KV heads
    x 128 values (2,359,296 vectors, 604 MB fp16, larger than L2).  Bytes per vector: 256 fp16 +
    128 codes + 2 scale, read and written once per direction."""
    n = 36 * 2 * 8 * 4096
    g = torch.Generator(device=dev).manual_seed(7700)
    kv = (torch.randn((n, 128), device=dev, generator=g) * 2.0).half()
    codes = torch.empty((n, 128), dtype=torch.int8, device=dev)
    scales = torch.empty(n, dtype=torch.float16, device=dev)
    back = torch.empty_like(kv)
    per_vec = 256 + 128 + 2
    hbm = load_peaks().get("hbm_gbs", 6800.0)
    out = {"workload": "KV cache of 4096 tokens, 36 layers x K,V x 8 heads x 128 (fp16 <-> int8 + fp16 scale "
                       "per head vector)", "vectors": n, "bytes_per_launch": n * per_vec}
    for name, fn in (("encode", lambda: q.jllm_kv_encode_i8(kv, codes=codes, scales=scales)),
                     ("decode", lambda: q.jllm_kv_decode_i8(codes, scales, out=back))):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            fn()
        torch.cuda.synchronize()
        t = time_graph(torch, gr, stream, max(10, args.steps // 2), 3)
        del gr
        gbs = n * per_vec / t / 1e9
        out[name] = {"us": round(t * 1e6, 1), "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm,
                                                           "unit": "GB/s", "frac": round(gbs / hbm, 4),
                                                           "kernel": f"kv_{name}_kernel"}}
    return out


def run_ffn_lmhead(torch, q, W, dev, stream, args):
    """Fused FFN block plus LM head: h = silu(x Wg^T) * (x Wu^T) (fp16, one pass), y = h Wd^T
    (fp32), logits = x Wlm^T (2560 -> 151936, fp32), at M = 1 (weight GB/s) and M = 512
    (TFLOP/s).  Gate/up/down are the first layer's weights of the sweep."""
    K, NF = 2560, 9728
    NL = synthetic.LM_HEAD[2]  # (name, K, N)
    wg, wu, wd = W[4], W[5], W[6]
    wlm = torch.from_numpy(synthetic.q4k_weights(NL, K, synthetic.weight_seed(4, 0, 7))).to(dev)
    wbytes = 2 * weight_bytes(NF, K) + weight_bytes(K, NF) + weight_bytes(NL, K)
    out = {}
    for M in (1, 512):
        x = torch.from_numpy(synthetic.activations(M, K, synthetic.activation_seed(4, M, 0))).to(dev)
        h = torch.empty((M, NF), dtype=torch.float16, device=dev)
        yd = torch.empty((M, K), dtype=torch.float32, device=dev)
        ylm = torch.empty((M, NL), dtype=torch.float32, device=dev)

        def step():
            q.jllm_q4k_ffn_swiglu(wg, wu, x, NF, K, out=h)
            q.jllm_q4k_gemm(wd, h, K, NF, out=yd)
            q.jllm_q4k_gemm(wlm, x, NL, K, out=ylm)

        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        torch.cuda.synchronize()
        t = time_graph(torch, g, stream, max(5, args.steps // 10), 3)
        del g
        flops = 2.0 * M * (2 * NF * K + K * NF + NL * K)
        pk = load_peaks()
        hbm, burst = pk.get("hbm_gbs", 6800.0), pk.get("bf16_tflops", 1900.0)
        gbs, tf = wbytes / t / 1e9, flops / t / 1e12
        # M = 1 streams the weights (HBM-bound); M = 512 is far above the balance point
        roof = ({"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                 "kernel": "q4k_gemv_kernel"} if M == 1 else
                {"bound": "tensor", "achieved": round(tf, 2), "peak": burst, "unit": "TFLOP/s",
                 "frac": round(tf / burst, 4), "kernel": "q4k_gemm_tc_kernel",
                 "peak_source": "measured bf16 burst (fp16 dense rate equal)"})
        out[f"M{M}"] = {"us_per_step": round(t * 1e6, 1), "weight_gbs": round(gbs, 1),
                        "tflops": round(tf, 2), "launches_per_step": 3, "roofline": roof}
        if M == 1:
            # the LM head alone: one large independent GEMV launch, the kernel's sustained rate
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                q.jllm_q4k_gemm(wlm, x, NL, K, out=ylm)
            torch.cuda.synchronize()
            tl = time_graph(torch, g, stream, max(5, args.steps // 10), 3)
            del g
            lb = weight_bytes(NL, K)
            peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
                os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
            hbm = peaks.get("hbm_gbs", 6800.0)
            out["lm_head_M1"] = {"us": round(tl * 1e6, 1), "weight_gbs": round(lb / tl / 1e9, 1),
                                 "frac_of_hbm": round(lb / tl / 1e9 / hbm, 4)}
    out["workload"] = ("ffn_swiglu 2560->2x9728 (fp16 h), down 9728->2560 (fp32), "
                       "LM head 2560->151936 (fp32); weight bytes %d per step" % wbytes)
    return out


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    return json.load(open(path)) if os.path.exists(path) else {}


def run_prefill(torch, q, W, meta, dev, stream, args, world, M=M_PREFILL, short=False, tmax=None, sync=None,
                light=False):
    """M = 2048 tcgen05 GEMMs over the same resident weights, fp16 out.  The value is
    the layer's data flow in four launches (q/k/v and gate/up each one batched GEMM
    on their shared X, then o, then down); the seven-call sweep is timed beside it.
    short=True: the short-prompt sizes (M = 33, 235) with per-token scaled X, each with
    the fraction of the bound that applies at that M (HBM below the balance point
    M* ~ 83, the tensor cores above).  light=True: the four-launch sweep alone (the
    other long-prompt sizes, M = 1024 and 3072)."""
    xs = {}
    for (_, K, N) in meta:
        if K not in xs:
            seed = synthetic.activation_seed(2 if short else 3, M, K)
            xs[K] = torch.from_numpy(synthetic.activations(M, K, seed, per_token_scale=short)).to(dev)
    # one output per shape of a layer (k and v must not share one inside a batch)
    ys = [torch.empty((M, N), dtype=torch.float16, device=dev) for (_, K, N) in meta[:len(SHAPES)]]
    flops = sum(2.0 * M * N * K for (_, K, N) in meta)
    layers = len(meta) // len(SHAPES)

    def sweep7():
        for i, (w, (_, K, N)) in enumerate(zip(W, meta)):
            q.jllm_q4k_gemm(w, xs[K], N, K, out=ys[i % len(SHAPES)])

    def sweep_batched():
        for layer in range(layers):
            base = layer * len(SHAPES)
            for _, members in GROUPS:
                K = meta[base + members[0]][1]
                if len(members) == 1:
                    i = members[0]
                    q.jllm_q4k_gemm(W[base + i], xs[K], meta[base + i][2], K, out=ys[i])
                else:
                    q.jllm_q4k_gemm_batch([W[base + i] for i in members], xs[K], [meta[base + i][2] for i in members],
                                          K, outs=[ys[i] for i in members])

    def timed(fn, clk=None):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        torch.cuda.synchronize()
        t = time_graph(torch, g, stream, max(2, args.steps // 5), max(3, args.warmup // 2), clk)
        del g
        return t

    peaks = load_peaks()
    burst = peaks.get("bf16_tflops", 1900.0)
    if short:
        t, t7 = timed(sweep_batched), timed(sweep7)
        wb = sum(weight_bytes(N, K) for (_, K, N) in meta)
        gbs, tf = wb / t / 1e9, flops / t / 1e12
        # balance point of the roofline: M* = 0.5625 B/weight * tensor peak / (2 * HBM peak)
        mstar = 0.5625 * burst * 1e12 / (2 * peaks.get("hbm_gbs", 6800.0) * 1e9)
        if M < mstar:
            roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks.get("hbm_gbs", 6800.0), "unit": "GB/s",
                    "frac": round(gbs / peaks.get("hbm_gbs", 6800.0), 4)}
        else:
            roof = {"bound": "tensor", "achieved": round(tf, 2), "peak": burst, "unit": "TFLOP/s",
                    "frac": round(tf / burst, 4)}
        kern = ("q4k_gemm_mma_kernel" if M <= 24 else
                "q4k_gemm_tc_kernel (gate/up) + q4k_gemm_mma_kernel (q/k/v, o, down)" if M <= 40 else
                "q4k_gemm_tc_kernel")
        roof.update({"balance_point_M": round(mstar, 1), "peak_source": "measured (burst bf16; fp16 dense rate equal)",
                     "kernel": kern})
        return {"M": M, "us_per_step": round(t * 1e6, 1), "weight_gbs": round(gbs, 1),
                "tflops": round(tf, 2), "launches_per_step": layers * len(GROUPS), "roofline": roof,
                "seven_call": {"us_per_step": round(t7 * 1e6, 1), "weight_gbs": round(wb / t7 / 1e9, 1),
                               "tflops": round(flops / t7 / 1e12, 2)}}
    if light:
        t = (tmax or (lambda v: v))(timed(sweep_batched))
        tf = flops / t / 1e12
        return {"M": M, "value": round(tf * world, 2), "unit": "TFLOP/s", "ms_per_step": round(t * 1e3, 3),
                "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": burst, "unit": "TFLOP/s",
                             "frac": round(tf / burst, 4), "peak_source": "measured bf16 burst (fp16 dense rate equal)",
                             "kernel": "q4k_gemm_tc_kernel"}}
    tmax = tmax or (lambda t: t)
    if sync:
        sync()
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        t = tmax(timed(sweep_batched, clk))
    if sync:
        sync()
    t7 = tmax(timed(sweep7))
    peak = burst
    tf = flops / t / 1e12
    return {"value": round(tf * world, 2), "unit": "TFLOP/s", "ms_per_step": round(t * 1e3, 3),
            "config": {"workload": f"prefill sweep M={M}, {layers} layers x 7 shapes in 4 launches per layer "
                                   "(qkv and gate/up batched), fp16 out",
                       "flops_per_step": flops, "launches_per_step": layers * len(GROUPS)},
            "prefill_7call": {"value": round(flops * world / t7 / 1e12, 2), "unit": "TFLOP/s",
                              "ms_per_step": round(t7 * 1e3, 3), "launches_per_step": len(meta)},
            "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(tf / peak, 4), "traffic": profiled_traffic("q4k_gemm_tc_kernel"),
                         "peak_source": "measured bf16 burst: the step is ~15 ms, not a seconds-long loop "
                                        "(fp16 dense rate equal)",
                         "frac_of_sustained": round(tf / peaks.get("bf16_tflops_sustained", 1700.0), 4),
                         "kernel": "q4k_gemm_tc_kernel"},
            "clocks": clk.summary()}


# ------------------------------------------------------------ CPU baseline --
def host_cpu():
    """CPU model and core count of this host (the oracle uses one core).  The model comes from
    lscpu ("Model name", which names Arm cores such as Neoverse-V2), else /proc/cpuinfo."""
    model, vendor = "", ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name" and not model:
                model = v.strip()
            elif k.strip() == "Vendor ID" and not vendor:
                vendor = v.strip()
    except Exception:
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                k = line.split(":")[0].strip().lower()
                if k in ("model name", "cpu model", "hardware") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    import platform

    name = " ".join(x for x in (vendor, model) if x) or platform.processor() or platform.machine()
    return {"model": name, "arch": platform.machine(), "nproc": os.cpu_count(),
            "used": "1 of %d cores" % (os.cpu_count() or 0)}


def cpu_baseline(budget_s=12.0):
    """The oracle (single-threaded fp64 C) on the first layers of the decode sweep, bounded in time."""
    import oracle

    oracle.build()
    done_bytes = 0
    t_total = 0.0
    layers = 0
    for layer in range(N_LAYERS):
        for idx, (name, K, N) in enumerate(SHAPES):
            w = synthetic.q4k_weights(N, K, synthetic.weight_seed(1, layer, idx))
            x = synthetic.activations(1, K, synthetic.activation_seed(1, layer * 8 + group_index(idx)))
            t0 = time.perf_counter()
            oracle.matmul(w, x, N, K)
            t_total += time.perf_counter() - t0
            done_bytes += weight_bytes(N, K)
        layers += 1
        if t_total >= budget_s:
            break
    return {"value": round(done_bytes / t_total / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"decode sweep, first {layers} of 36 layers x 7 shapes ({done_bytes} weight bytes), "
                      f"{t_total:.1f} s single-threaded fp64",
            "host": host_cpu()}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle

    oracle.build()
    # each step: one layer of the decode sweep (7 shapes), cycling layers
    per_step_bytes = sum(weight_bytes(N, K) for (_, K, N) in SHAPES)
    inputs = []
    n_layers = min(N_LAYERS, args.warmup + args.steps)
    for layer in range(n_layers):
        inputs.append([(synthetic.q4k_weights(N, K, synthetic.weight_seed(1, layer, idx)),
                        synthetic.activations(1, K, synthetic.activation_seed(1, layer * 8 + group_index(idx))), N, K)
                       for idx, (_, K, N) in enumerate(SHAPES)])

    def step(i):
        for w, x, N, K in inputs[i % n_layers]:
            oracle.matmul(w, x, N, K)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    t = (time.perf_counter() - t0) / args.steps
    v = per_step_bytes / t / 1e9
    line = {
        "impl": "reference",
        "metric": "Q4_K matmul: M=1 weight GB/s vs HBM peak; M=2048 TFLOP/s vs BF16 peak",
        "value": round(v, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded GGUF Q4_K blocks, fp16 N(0,1) activations)",
        "config": {"workload": "decode sweep M=1, one layer (7 Qwen3-4B shapes) per step, single-threaded CPU oracle"},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} layers of the decode sweep, one per step", "host": host_cpu()},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_tc_rates(args):
    """Sustained tensor-core rates on one GPU, for the int8 ("MMQ") question: tcgen05.mma
    kind::f16 (the GEMM's instruction) against the warp-level mma.sync f16 and s8 instructions
    (tcgen05.mma kind::i8 does not assemble for sm_103a).  Operands resident, zero-valued;
    CUDA events around each launch."""
    import ctypes

    import torch

    import __graft_entry__

    lib = ctypes.CDLL(__graft_entry__._load_builder().build_microbench())
    lib.jllm_microbench_tc_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p]
    lib.jllm_microbench_tc_rate.restype = ctypes.c_int
    dev = torch.device("cuda", 0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = torch.cuda.Stream()
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    out = {"sms": sms}
    # (kind, name, CTAs, warps per CTA measured, ops per instruction, instructions per iteration per issuer)
    cases = ((0, "tcgen05_kind_f16", sms, 1, 2 * 128 * 256 * 16, 4),
             (1, "mma_sync_f16_m16n8k16", 2 * sms, 8, 2 * 16 * 8 * 16, 4),
             (2, "mma_sync_s8_m16n8k32", 2 * sms, 8, 2 * 16 * 8 * 32, 4),
             # the tcgen05 stream with a commit per 4 MMAs, and a probe of a completed barrier phase
             (5, "tcgen05_kind_f16_commit_per_4", sms, 1, 2 * 128 * 256 * 16, 4),
             (3, "tcgen05_kind_f16_commit_try_wait_per_4", sms, 1, 2 * 128 * 256 * 16, 4),
             (4, "tcgen05_kind_f16_commit_test_wait_per_4", sms, 1, 2 * 128 * 256 * 16, 4))
    for kind, name, ctas, wpc, ops, per_iter in cases:
        cyc = torch.zeros(ctas * wpc, dtype=torch.int64, device=dev)
        best = None
        for iters in (2000, 20000, 20000):
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            start.record(stream)
            rc = lib.jllm_microbench_tc_rate(kind, ctas, iters, cyc.data_ptr(), sink.data_ptr(), stream.cuda_stream)
            end.record(stream)
            end.synchronize()
            if rc != 0:
                raise RuntimeError(f"{name}: microbench returned {rc}")
            t = start.elapsed_time(end) / 1e3
            rate = ctas * wpc * iters * per_iter * ops / t / 1e12
            best = max(best or 0.0, rate)
        c = cyc.double()
        out[name] = {"tops": round(best, 1), "cycles_per_instr_per_issuer": round(float(c.max()) / (20000 * per_iter), 2)}
    out["tcgen05_kind_i8"] = "not available: ptxas (CUDA 13.0) rejects tcgen05.mma .kind::i8 for sm_103a"
    peaks = load_peaks()
    out["measured_cublas_bf16_tflops"] = peaks.get("bf16_tflops")
    print(json.dumps({"tc_rates": out}), flush=True)


def main():
    args = parse()
    if args.tc_rates:
        run_tc_rates(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
