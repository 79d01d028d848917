#!/usr/bin/env python3
"""Benchmark of the quantized GCN message-passing layer on GB300.

One step = the whole hot path over the 3-layer GCN workload (R-MAT graph,
131,072 nodes, 128 -> 256 -> 256 -> 47, 40% marginal nodes): for each
message bit-width b in (2, 4, 8), one forward and one backward pass of the
three layers (quantize, de-quantizing aggregation, tcgen05 update GEMM,
and their backward), i.e. the three runs of that workload.

Metric: layer-edges per second, fwd+bwd.  Each layer's forward+backward
counts the graph's E edges (self-loops included) once:
    value = 3 layers x 3 runs x E / step time.

Usage:
  python bench.py [--steps K] [--warmup W] [--impl ours|reference]
  torchrun --nproc-per-node N bench.py --gpus N   (N independent replicas)

Prints one JSON line (rank 0).  Timing: CUDA events on the launching
stream around each step, L2 flushed (a 256 MiB write) between steps.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth.configs import BY_NAME, GCN3_RMAT17  # noqa: E402

METRIC = "GNN layer edges/sec fwd+bwd at 1 GB300; quantized SpMM HBM GB/s vs peak"
UNIT = "edges/s"
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device) -> float:
    """The largest x over all ranks: a job's time is its slowest rank's."""
    if ws <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: float, ws: int, ms_per_step: float) -> float:
    """Whole-job units per second: every rank processes its own units in the
    same (slowest-rank) time."""
    return units_per_rank_step * ws / (ms_per_step / 1e3)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while the
    timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # the timed region starts once the sampler is live
            t0 = time.perf_counter()
            while not self.lines and self.proc.poll() is None and time.perf_counter() - t0 < 5.0:
                time.sleep(0.02)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=5)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def make_inputs(w, device):
    g = w.make_graph(device=device)
    widths = w.widths
    X = synth.normal_matrix(g.n, widths[0], seed=w.seed, device=device)
    Ws = [synth.glorot(widths[l], widths[l + 1], seed=w.seed + 1 + l, device=device) for l in range(len(widths) - 1)]
    mask = synth.bernoulli_mask(g.n, w.mask_frac, seed=w.seed, device=device)
    dY = synth.normal_matrix(g.n, widths[-1], seed=w.seed, tag=synth.TAG_GRAD, device=device)
    return g, X, Ws, mask, dY


def seeds_for(base, L, b):
    f = [synth.layer_seed(base ^ (b << 56), l, False) for l in range(L)]
    bw = [synth.layer_seed(base ^ (b << 56), l, True) for l in range(L)]
    return f, bw


def spmm_bytes(n, nnz, d, bits, n_marg, rows_gathered_marg, out_elem_bytes, q):
    """Algorithmic bytes of one de-quantizing aggregation.
    compulsory: every array once (each gathered message row read once);
    streaming: every edge's gathered row counted."""
    pitch = q.packed_pitch(d, bits) if bits < 32 else 0
    meta = (n + 1) * 4 + nnz * 4 + 2 * n * 4 + (n if bits < 32 else 0)
    out = n * d * out_elem_bytes
    comp = meta + n_marg * pitch + (n - n_marg) * d * 4 + out
    stream = (n + 1) * 4 + nnz * 4 * 2 + (nnz if bits < 32 else 0) + n * 4 + out \
        + rows_gathered_marg * pitch + (nnz - rows_gathered_marg) * d * 4
    return comp, stream


# --------------------------------------------------------------------------
# CPU oracle leg
# --------------------------------------------------------------------------

def oracle_layer_inputs(w, g, device="cpu"):
    """Inputs of the bounded CPU sample: the workload's middle layer
    (widths[1] -> widths[2]) with a synthetic post-ReLU input."""
    d_in, d_out = w.widths[1], w.widths[2]
    H = torch.relu(synth.normal_matrix(g.n, d_in, seed=w.seed + 11, device=device))
    W = synth.glorot(d_in, d_out, seed=w.seed + 12, device=device)
    dY = synth.normal_matrix(g.n, d_out, seed=w.seed + 13, tag=synth.TAG_GRAD, device=device)
    return H, W, dY


def oracle_layer_step(orc, rp, co, H, W, mask, bits, seed, dY):
    """The oracle's forward + backward of one hidden GCN layer (ReLU)."""
    sf, sb = synth.layer_seed(seed, 1, False), synth.layer_seed(seed, 1, True)
    o = orc.gcn_layer_fwd(rp, co, orc.COEF_GCN, H, W, mask, bits, sf, relu=True)
    orc.gcn_layer_bwd(rp, co, orc.COEF_GCN, dY, o["A"], o["Z"], W, mask, bits, sb, relu=True, need_dinput=True)


def _sample_text(w, g, bits):
    return (f"one hidden layer ({w.widths[1]} -> {w.widths[2]}, ReLU) forward+backward per step on the whole "
            f"graph ({g.n} nodes, {g.nnz} edges), b = {bits}, {int(w.mask_frac * 100)}% marginal, float64 oracle; "
            f"edges/s = E / time of that layer")


def run_reference(args, w):
    """The oracle as it stands, on the host cores."""
    import oracle
    oracle.build()
    g = w.make_graph()
    mask = synth.bernoulli_mask(g.n, w.mask_frac, seed=w.seed).numpy()
    H, W, dY = (x.numpy() for x in oracle_layer_inputs(w, g))
    rp, co = g.rowptr.numpy(), g.col.numpy()
    bits_cycle = list(w.bits)
    for i in range(args.warmup):
        oracle_layer_step(oracle, rp, co, H, W, mask, bits_cycle[i % len(bits_cycle)], w.seed, dY)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_layer_step(oracle, rp, co, H, W, mask, bits_cycle[i % len(bits_cycle)], w.seed, dY)
    dt = time.perf_counter() - t0
    value = args.steps * g.nnz / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "nodes": g.n, "edges": g.nnz,
                                            "widths": list(w.widths), "bits": list(w.bits)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": _sample_text(w, g, bits_cycle)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(w, g, mask):
    """Time the oracle on a bounded sample of the same workload."""
    import oracle
    oracle.build()
    rp, co = g.rowptr.cpu().numpy(), g.col.cpu().numpy()
    H, W, dY = (x.numpy() for x in oracle_layer_inputs(w, g))
    b = w.bits[0]
    t0 = time.perf_counter()
    oracle_layer_step(oracle, rp, co, H, W, mask.cpu().numpy(), b, w.seed, dY)
    dt = time.perf_counter() - t0
    return {"value": g.nnz / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": _sample_text(w, g, b) + f"; {dt:.1f} s"}


# --------------------------------------------------------------------------
# GPU leg
# --------------------------------------------------------------------------

def run_ours(args, w):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import quantized_gnn_message_gb300 as q
    from quantized_gnn_message_gb300.build import build
    from quantized_gnn_message_gb300.model import BWD_STAGES, FWD_STAGES, GCNStack
    build()
    q.lib()

    g, X, Ws, mask, dY = make_inputs(w, dev)
    G = q.graph_prepare(g.rowptr, g.col)
    model = GCNStack(G, w.widths, mask)
    L = model.L
    bits_list = list(w.bits)
    seeds = {b: seeds_for(w.seed, L, b) for b in bits_list}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step(events=None):
        for i, b in enumerate(bits_list):
            sf, sb = seeds[b]
            ef = None if events is None else events[i][0]
            eb = None if events is None else events[i][1]
            model.forward(X, Ws, b, sf, events=ef)
            model.backward(dY, Ws, b, sb, events=eb)

    def new_events():
        out = []
        for _ in bits_list:
            ef = [[_ev() for _ in range(2 * len(FWD_STAGES))] for _ in range(L)]
            eb = [[_ev() for _ in range(2 * len(BWD_STAGES))] for _ in range(L)]
            out.append((ef, eb))
        return out

    def _ev():
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        return e

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()

    stage_events = [new_events() for _ in range(args.steps)]
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        torch.cuda.profiler.start()  # an ncu --profile-from-start off capture sees the timed steps only
        for k in range(args.steps):
            flush.fill_(k & 0xFF)
            starts[k].record()
            step(stage_events[k])
            ends[k].record()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
    if int(model.err.item()) != 0:
        raise RuntimeError(f"device wait timed out (code {int(model.err.item())})")
    step_ms = [starts[k].elapsed_time(ends[k]) for k in range(args.steps)]
    total_ms = max_over_ranks(sum(step_ms), ws, dev)
    ms_per_step = total_ms / args.steps
    edges_per_step = L * len(bits_list) * g.nnz
    value = job_throughput(edges_per_step, ws, ms_per_step)

    # per-stage device time, from the events recorded inside the timed steps
    stage_ms = {}
    for k in range(args.steps):
        for i, b in enumerate(bits_list):
            ef, eb = stage_events[k][i]
            for l in range(L):
                for s, name in enumerate(FWD_STAGES):
                    stage_ms.setdefault((name, l, b), []).append(ef[l][2 * s].elapsed_time(ef[l][2 * s + 1]))
                for s, name in enumerate(BWD_STAGES):
                    if name in ("da_gemm", "quantize_bwd", "aggregate_t") and l == 0:
                        continue
                    stage_ms.setdefault((name, l, b), []).append(eb[l][2 * s].elapsed_time(eb[l][2 * s + 1]))

    # dominant kernel: the de-quantizing aggregation (forward + transposed)
    mk = mask.to(torch.int64)
    outdeg = torch.bincount(g.col.long(), minlength=g.n)
    indeg = (g.rowptr[1:] - g.rowptr[:-1]).long()
    n_marg = int(mk.sum().item())
    marg_out = int((outdeg * mk).sum().item())   # gathered marginal rows, forward
    marg_in = int((indeg * mk).sum().item())     # gathered marginal rows, transposed
    agg_bytes_c, agg_bytes_s, agg_ms, agg_launches = 0, 0, 0.0, 0
    for (name, l, b), times in stage_ms.items():
        if name not in ("aggregate", "aggregate_t"):
            continue
        d = w.widths[l]
        fwd = name == "aggregate"
        c, s_ = spmm_bytes(g.n, g.nnz, d, b, n_marg, marg_out if fwd else marg_in, 2 if fwd else 4, q)
        agg_bytes_c += c * len(times)
        agg_bytes_s += s_ * len(times)
        agg_ms += sum(times)
        agg_launches += len(times)
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = agg_bytes_c / (agg_ms / 1e3) / 1e9
    traffic = load_traffic(w.name)
    stage_summary = {}
    for (name, l, b), times in stage_ms.items():
        stage_summary.setdefault(name, 0.0)
        stage_summary[name] += sum(times) / args.steps
    roofline = {"kernel": "spmm_bulk_kernel (de-quantizing aggregation, forward and transposed)",
                "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"hbm_gbs of {peak_kind}",
                "traffic": traffic,
                "algorithmic_bytes_per_launch": agg_bytes_c / max(agg_launches, 1),
                "streaming_bytes_per_launch": agg_bytes_s / max(agg_launches, 1),
                "avg_launch_ms": agg_ms / max(agg_launches, 1)}

    # end to end through the public API: pinned host inputs in, dW out
    Xh = X.cpu().pin_memory()
    dYh = dY.cpu().pin_memory()
    dW_host = [torch.empty(x.shape, dtype=torch.float32).pin_memory() for x in model.dW]
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    h2d = Xh.numel() * 4 + dYh.numel() * 4
    d2h = sum(x.numel() * 4 for x in dW_host) * len(bits_list)
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        e_s[k].record()
        X.copy_(Xh, non_blocking=True)
        dY.copy_(dYh, non_blocking=True)
        for b in bits_list:
            sf, sb = seeds[b]
            model.forward(X, Ws, b, sf)
            model.backward(dY, Ws, b, sb)
            for hw, dw in zip(dW_host, model.dW):
                hw.copy_(dw, non_blocking=True)
        e_e[k].record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(e_s[k].elapsed_time(e_e[k]) for k in range(args.steps)) / args.steps, ws, dev)
    e2e = {"value": job_throughput(edges_per_step, ws, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    launches = sum(model.launches(b) for b in bits_list) * args.steps
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "arithmetic": "f32 accumulation; 2/4/8-bit message codes; bf16 tensor-core GEMM inputs",
            "data": "synthetic",
            "config": {"workload": w.name, "nodes": g.n, "edges": g.nnz, "widths": list(w.widths),
                       "bits": bits_list, "marginal_fraction": w.mask_frac, "coefficients": "gcn",
                       "l2": "flushed (256 MiB write) before every timed step",
                       "parallelism": "replicas" if ws > 1 else "single"},
            "roofline": roofline,
            "stage_ms_per_step": {k: round(v, 4) for k, v in stage_summary.items()},
            "e2e": e2e, "gpu_launches": launches}
    cs = clocks.summary()
    if cs is not None:
        line["clocks"] = cs
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, g.to("cpu"), mask)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def _timed(fn, iters, flush):
    """Average device ms of fn() over `iters` calls, L2 flushed before each,
    after one untimed call (module loading, first workspace allocation)."""
    fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for a, b in evs:
        flush.fill_(1)
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / iters


def run_gat(args, w):
    """GAT layer forward+backward (Tango Fig. 1a/1b) on one GPU."""
    import quantized_gnn_message_gb300 as q
    from quantized_gnn_message_gb300.build import build
    build()
    q.lib()
    dev = torch.device("cuda", 0)
    if args.graph_scale is not None:
        import dataclasses
        S = args.graph_scale
        w = dataclasses.replace(w, name=f"gat-rmat{S}", graph=dict(kind="rmat", scale=S, n=1 << S,
                                                                   n_draws=16 << S, exact_edges=16 << S))
    g = w.make_graph(device=dev)
    d_in, heads, f = w.widths
    d = heads * f
    G = q.graph_prepare(g.rowptr, g.col)
    H = synth.normal_matrix(g.n, d_in, seed=w.seed, device=dev)
    Wt = synth.glorot(d_in, d, seed=w.seed + 1, device=dev)
    a_s = synth.glorot(heads, f, seed=w.seed + 2, device=dev)
    a_d = synth.glorot(heads, f, seed=w.seed + 3, device=dev)
    dOut = synth.normal_matrix(g.n, d, seed=w.seed, tag=synth.TAG_GRAD, device=dev)
    bits = w.bits[0]
    L = q.GATLayer(G, d_in, heads, f, 0.2, bits, None, alpha_bits=args.alpha_bits)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    fwd = lambda: L.forward(H, Wt, a_s, a_d, 1)
    bwd = lambda: L.backward(dOut, H, Wt, a_s, a_d, 2)
    for _ in range(args.warmup):
        fwd()
        bwd()
    with ClockSampler(0) as clocks:
        torch.cuda.profiler.start()
        t_f = _timed(fwd, args.steps, flush)
        t_b = _timed(bwd, args.steps, flush)
        torch.cuda.profiler.stop()
    # dominant edge kernels alone, same inputs
    t_sm = _timed(lambda: q.sddmm_edge_softmax(G, L.S, L.D), args.steps, flush)
    out = torch.empty(g.n, d, device=dev)
    t_sp = _timed(lambda: q.edge_spmm(G, L.alpha, L.Hp, None, None, d, 32, out=out), args.steps, flush)
    # the 8-bit attention path (Tango Sec. 3.3): quantizer and SpMM over the codes
    codes, hdr = q.quantize_edge_values(G, L.alpha, 1)
    t_aq = _timed(lambda: q.quantize_edge_values(G, L.alpha, 1), args.steps, flush)
    t_sp8 = _timed(lambda: q.edge_spmm_alpha8(G, codes, hdr, L.Hp, None, None, d, 32, out=out), args.steps, flush)
    E, n = g.nnz, g.n
    sm_bytes = (n + 1) * 4 + E * 4 + 2 * n * heads * 4 + E * heads * 4
    sp_bytes = (n + 1) * 4 + E * 4 + E * heads * 4 + n * d * 4 * 2
    aq_bytes = (n + 1) * 4 + E * heads * 4 + E * heads + n * heads * 8
    sp8_bytes = (n + 1) * 4 + E * 4 + E * heads + n * heads * 8 + n * d * 4 * 2
    peaks, kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    step_ms = t_f + t_b
    line = {"metric": METRIC, "value": E / (step_ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32",
            "arithmetic": "f32 accumulation; bf16 tensor-core GEMM inputs", "data": "synthetic",
            "config": {"workload": w.name, "nodes": n, "edges": E, "d_in": d_in, "heads": heads, "f": f,
                       "bits": bits, "alpha_bits": args.alpha_bits, "l2": "flushed before every timed call"},
            "stages_ms": {"layer_fwd": t_f, "layer_bwd": t_b, "edge_softmax": t_sm, "edge_spmm": t_sp,
                          "alpha_quantize": t_aq, "edge_spmm_alpha8": t_sp8},
            "kernels_gbs": {"edge_softmax": sm_bytes / (t_sm / 1e3) / 1e9,
                            "edge_spmm": sp_bytes / (t_sp / 1e3) / 1e9,
                            "alpha_quantize": aq_bytes / (t_aq / 1e3) / 1e9,
                            "edge_spmm_alpha8": sp8_bytes / (t_sp8 / 1e3) / 1e9},
            "roofline": {"kernel": "edge_spmm_kernel (multi-head aggregation)", "bound": "hbm",
                         "achieved": sp_bytes / (t_sp / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": sp_bytes / (t_sp / 1e3) / 1e9 / peak, "peak_source": f"hbm_gbs of {kind}",
                         "traffic": None, "algorithmic_bytes_per_launch": sp_bytes, "avg_launch_ms": t_sp}}
    cs = clocks.summary()
    if cs is not None:
        line["clocks"] = cs
    print(json.dumps(line), flush=True)


def run_aggregate(args, w):
    """Quantize + de-quantizing aggregation forward + transposed, alone, over
    a sweep of widths and bit-widths (all nodes marginal)."""
    import quantized_gnn_message_gb300 as q
    from quantized_gnn_message_gb300.build import build
    build()
    q.lib()
    dev = torch.device("cuda", 0)
    if args.graph_scale is not None:
        import dataclasses
        S = args.graph_scale
        w = dataclasses.replace(w, name=f"aggregate-rmat{S}",
                                graph=dict(kind="rmat", scale=S, n=1 << S, n_draws=32 << S))
    t0 = time.perf_counter()
    g = w.make_graph(device=dev)
    t_gen = time.perf_counter() - t0
    t0 = time.perf_counter()
    G = q.graph_prepare(g.rowptr, g.col)
    torch.cuda.synchronize()
    t_prep = time.perf_counter() - t0
    ds = [int(x) for x in args.sweep_d.split(",")] if args.sweep_d else list(w.sweep_d)
    bl = [int(x) for x in args.sweep_bits.split(",")] if args.sweep_bits else list(w.bits)
    dmax = max(ds)
    X = synth.normal_matrix(g.n, dmax, seed=w.seed, device=dev)
    Y = torch.empty(g.n * dmax, dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    E, n = g.nnz, g.n
    peaks, kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    L = q.lib()
    rows = []
    tot_edges, tot_ms = 0, 0.0
    best = None
    beta_rows = []
    bt = torch.empty(n, dtype=torch.float32, device=dev)
    with ClockSampler(0) as clocks:
        for d in ds:
            Xd = X[:, :d]
            Yd = Y[:n * d].view(n, d)
            tbeta = _timed(lambda: q.message_variance_weights(G, Xd, q.COEF_GCN, out=bt), args.steps, flush)
            bbytes = n * d * 4 + (n + 1) * 4 + E * 4 + n * 4 + n * 4
            beta_rows.append({"d": d, "beta_ms": tbeta, "beta_gbs": bbytes / (tbeta / 1e3) / 1e9})
            # AdaQP's per-message width choice from beta (Problems 10-12 on one device)
            rbt = torch.empty(n, dtype=torch.uint8, device=dev)
            tab = _timed(lambda: q.assign_bits(bt, d, 0.5, 1e-3, out=rbt), args.steps, flush)
            beta_rows[-1].update({"assign_bits_ms": tab, "assign_bits_gbs": n * 5 / (tab / 1e3) / 1e9})
            del rbt
            if d <= 256 and d % 4 == 0:
                # per-message widths drawn uniformly from {2, 4, 8} (AdaQP's sampling ablation)
                u = synth.uniform01(synth.stream_seed(w.seed, 0x42), torch.arange(n, dtype=torch.int64, device=dev), 0)
                rb = torch.tensor([2, 4, 8], dtype=torch.uint8, device=dev)[torch.clamp((u * 3).long(), max=2)]
                pkm, roff = q.quantize_pack_mixed(Xd, rb, 7)
                tmq = _timed(lambda: q.quantize_pack_mixed(Xd, rb, 7, roff=roff), args.steps, flush)
                tmf = _timed(lambda: q.dequant_spmm_mixed(G, Xd, pkm, roff, rb, out=Yd), args.steps, flush)
                mbytes = (n + 1) * 4 + E * 4 + 2 * n * 4 + n + n * 8 + int(roff[n].item()) + n * d * 4
                beta_rows[-1].update({"mixed_quantize_ms": tmq, "mixed_fwd_ms": tmf,
                                      "mixed_fwd_gbs_compulsory": mbytes / (tmf / 1e3) / 1e9,
                                      "mixed_edges_per_s": E / (tmf / 1e3)})
                del pkm, roff, rb, u
            for b in bl:
                pk = torch.empty(n, q.packed_pitch(d, b), dtype=torch.uint8, device=dev)
                qz = lambda: q.quantize_pack(Xd, None, b, 7, out=pk)
                qe = lambda: q.quant_error(Xd, pk, None, b)
                fw = lambda: q.dequant_spmm(G, None, pk, None, d, b, out=Yd)
                bw = lambda: q.dequant_spmm(G, None, pk, None, d, b, transpose=True, out=Yd)
                for _ in range(args.warmup):
                    qz(); fw(); bw()
                torch.cuda.profiler.start()
                tq = _timed(qz, args.steps, flush)
                tf = _timed(fw, args.steps, flush)
                tb = _timed(bw, args.steps, flush)
                te = _timed(qe, args.steps, flush)
                torch.cuda.profiler.stop()
                pitch = q.packed_pitch(d, b)
                comp = (n + 1) * 4 + E * 4 + 2 * n * 4 + n * pitch + n * d * 4
                stream = (n + 1) * 4 + E * 8 + n * 4 + E * pitch + n * d * 4
                qbytes = n * d * 4 + n * pitch
                r = {"d": d, "bits": b, "quantize_ms": tq, "fwd_ms": tf, "bwd_ms": tb,
                     "quantize_gbs": qbytes / (tq / 1e3) / 1e9,
                     "error_metric_ms": te, "error_metric_gbs": qbytes / (te / 1e3) / 1e9,
                     "fwd_gbs_compulsory": comp / (tf / 1e3) / 1e9, "bwd_gbs_compulsory": comp / (tb / 1e3) / 1e9,
                     "fwd_gbs_streaming": stream / (tf / 1e3) / 1e9, "bwd_gbs_streaming": stream / (tb / 1e3) / 1e9,
                     "edges_per_s_fwd": E / (tf / 1e3)}
                rows.append(r)
                tot_edges += 2 * E
                tot_ms += tf + tb
                if best is None or r["fwd_gbs_compulsory"] > best["fwd_gbs_compulsory"]:
                    best = r
                del pk
    line = {"metric": METRIC, "value": tot_edges / (tot_ms / 1e3), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "arithmetic": "f32 accumulation; 2/4/8-bit message codes",
            "data": "synthetic",
            "config": {"workload": w.name, "nodes": n, "edges": E, "sweep_d": ds, "bits": bl,
                       "generation_s": t_gen, "prepare_s": t_prep, "l2": "flushed before every timed call"},
            "sweep": rows, "per_width": beta_rows,
            "roofline": {"kernel": "spmm_kernel forward (best of sweep)", "bound": "hbm",
                         "achieved": best["fwd_gbs_compulsory"], "peak": peak, "unit": "GB/s",
                         "frac": best["fwd_gbs_compulsory"] / peak, "peak_source": f"hbm_gbs of {kind}",
                         "traffic": None, "at": {"d": best["d"], "bits": best["bits"]}}}
    cs = clocks.summary()
    if cs is not None:
        line["clocks"] = cs
    print(json.dumps(line), flush=True)


def load_traffic(workload):
    """DRAM traffic per launch of the aggregation kernel from the committed
    ncu summary, if it was taken on the kernel source as it is now."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    from quantized_gnn_message_gb300.build import AGGREGATION_SOURCES, source_digest
    ent = rec.get(workload)
    if not ent or ent.get("source_digest") != source_digest(AGGREGATION_SOURCES):
        return None
    return ent.get("dram_bytes_per_launch")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=GCN3_RMAT17.name, choices=list(BY_NAME))
    ap.add_argument("--sweep-d", default=None, help="aggregate workload: comma-separated widths")
    ap.add_argument("--sweep-bits", default=None, help="aggregate workload: comma-separated bit-widths")
    ap.add_argument("--graph-scale", type=int, default=None,
                    help="aggregate / GAT workloads: R-MAT scale S (2^S nodes; 32 / 16 draws per node) for smaller cases")
    ap.add_argument("--alpha-bits", type=int, default=32, choices=[32, 8],
                    help="GAT workload: 8 quantizes the attention values the SpMM reads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    w = BY_NAME[args.workload]
    if args.impl == "reference":
        ws, rank, _ = dist_env()
        if rank == 0:
            if w.kind != "gcn":
                print(json.dumps({"impl": "reference", "unavailable": "the oracle sample covers the GCN workloads"}))
            else:
                run_reference(args, w)
        return
    if w.kind != "gcn" and dist_env()[0] > 1 and dist_env()[1] != 0:
        return  # the GAT and sweep workloads run on one GPU (rank 0); their lines say n_gpus 1
    if w.kind == "gat":
        run_gat(args, w)
    elif w.kind == "aggregate":
        run_aggregate(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
