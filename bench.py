#!/usr/bin/env python3
"""Benchmark of the quantized GCN message-passing layer on GB300.

One step = the whole hot path over the large power-law GCN workload (R-MAT
graph with ogbn-products' counts: 2,449,029 nodes, 61,859,140 edges plus a
self-loop per node; widths 100 -> 256 -> 256 -> 47; 60% of the nodes
marginal, their messages quantized at 2 bits): one forward and one backward
pass of the three layers (quantize, de-quantizing aggregation, tcgen05
update GEMM, and their backward).

Metric: layer-edges per second, fwd+bwd.  Each layer's forward+backward
counts the graph's E edges (self-loops included) once:
    value = 3 layers x E / step time.

The same line carries the roofline of the dominant kernel (the
de-quantizing aggregation, forward and transposed, on this workload) and a
second record, `roofline_largest`, for the aggregation alone on the largest
graph (R-MAT, 16,777,216 nodes, ~537M edges, d = 256, b = 8, every row
packed), forward and transposed, timed with CUDA events.

Usage:
  python bench.py [--steps K] [--warmup W] [--impl ours|reference]
  torchrun --nproc-per-node N bench.py --gpus N   (N independent replicas)

Prints one JSON line (rank 0).  Timing: CUDA events on the launching
stream around each step; the inputs are larger than L2, and L2 is also
flushed (a 256 MiB write) between steps.
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
from synth.configs import AGG_SWEEP, BY_NAME, GCN3_LARGE  # noqa: E402

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


def spmm_bytes(n, nnz, d, bits, n_marg, rows_gathered_marg, out_elem_bytes, q, gated=False):
    """Algorithmic bytes of one de-quantizing aggregation.
    compulsory: every array once (each gathered message row read once);
    streaming: every edge's gathered row counted.  gated: the output goes
    through a ReLU gate read as bits (ceil(d / 32) words per row)."""
    pitch = q.packed_pitch(d, bits) if bits < 32 else 0
    meta = (n + 1) * 4 + nnz * 4 + 2 * n * 4 + (n if bits < 32 else 0)
    out = n * d * out_elem_bytes + (n * ((d + 31) // 32) * 4 if gated else 0)
    comp = meta + n_marg * pitch + (n - n_marg) * d * 4 + out
    stream = (n + 1) * 4 + nnz * 4 * 2 + (nnz if bits < 32 else 0) + n * 4 + out \
        + rows_gathered_marg * pitch + (nnz - rows_gathered_marg) * d * 4
    return comp, stream


# --------------------------------------------------------------------------
# CPU oracle leg
# --------------------------------------------------------------------------
#
# The oracle on the whole large graph takes minutes per layer, so both the
# CPU baseline and the reference arm time it on a stated row subset and
# scale each stage linearly by its own units:
#   - a seeded draw of R destination rows keeps all their in-edges;
#   - the sample graph holds those rows and every source they read,
#     renumbered 0..n'-1 (rows outside the draw have no in-edges);
#   - one step runs the workload's layer stack forward and backward on it,
#     stage by stage with the oracle's own routines (quantize, messages,
#     aggregation, GEMM, transposed aggregation), each stage timed;
#   - a stage's time is scaled by (its units on the whole graph) / (its
#     units in the sample): edges for the two aggregations, quantized rows
#     for the quantizer, rows for the GEMMs and the element-wise steps.
# The value is 3 layers x E over the scaled step time.

ORACLE_ROWS = 8000      # destination rows drawn per sampled step


class OracleSample:
    """The bounded CPU sample of a GCN workload (see above)."""

    def __init__(self, w, g, mask, rows=ORACLE_ROWS, seed=0):
        import numpy as np
        self.w = w
        rp = g.rowptr.cpu().numpy().astype(np.int64)
        co = g.col.cpu().numpy()
        mk = mask.cpu().numpy()
        n = g.n
        rng = np.random.default_rng(seed)
        R = np.sort(rng.choice(n, size=min(rows, n), replace=False))
        starts, ends = rp[R], rp[R + 1]
        eids = np.concatenate([np.arange(a, b) for a, b in zip(starts, ends)])
        nodes = np.union1d(R, co[eids])
        pos = {int(v): i for i, v in enumerate(nodes)}
        deg = np.zeros(nodes.size, np.int64)
        ridx = np.searchsorted(nodes, R)
        deg[ridx] = ends - starts
        srp = np.zeros(nodes.size + 1, np.int64)
        srp[1:] = np.cumsum(deg)
        scol = np.searchsorted(nodes, co[eids]).astype(np.int32)  # per row in CSR order, sources ascending
        self.rp, self.col = srp.astype(np.int32), scol
        self.nodes = nodes
        self.mask = mk[nodes]
        self.n_full, self.e_full = n, g.nnz
        self.m_full = int(mk.sum())
        self.e = int(eids.size)
        self.nn = int(nodes.size)
        self.mm = int(self.mask.sum())
        self.n_rows = int(R.size)
        del pos

    def inputs(self, X_full, dY_full):
        """The sample's rows of the workload's features and upstream gradient
        (torch tensors on any device), and its weights, as numpy arrays."""
        w = self.w
        idx = torch.from_numpy(self.nodes).to(X_full.device)
        X = X_full[idx].cpu().numpy()
        dY = dY_full[idx].cpu().numpy()
        Ws = [synth.glorot(w.widths[l], w.widths[l + 1], seed=w.seed + 1 + l).numpy()
              for l in range(len(w.widths) - 1)]
        return X, Ws, dY

    def step(self, orc, X, Ws, dY, bits, base_seed):
        """One forward + backward of the layer stack on the sample; returns
        the scaled whole-graph time (s) and the sample's wall time (s)."""
        import numpy as np
        L = len(Ws)
        scale = {"q": self.m_full / max(self.mm, 1), "e": self.e_full / max(self.e, 1),
                 "r": self.n_full / self.nn}
        t = {"q": 0.0, "e": 0.0, "r": 0.0}
        t_all = time.perf_counter()

        def timed(kind, f, *a, **k):
            t0 = time.perf_counter()
            r = f(*a, **k)
            t[kind] += time.perf_counter() - t0
            return r

        sf, sb = seeds_for(base_seed, L, bits)
        H = X
        saved = []
        for l in range(L):
            d = H.shape[1]
            pk = timed("q", orc.quantize, H, self.mask, bits, sf[l]) if bits < 32 else None
            M = timed("r", orc.messages, H, pk, self.mask, d, bits)
            A = timed("e", orc.spmm, self.rp, self.col, orc.COEF_GCN, M)
            Z = timed("r", orc.gemm, A, Ws[l], True)
            Hn = timed("r", lambda z: np.maximum(z, 0.0) if l < L - 1 else z, Z)
            saved.append((A, Z))
            H = Hn.astype(np.float32)
        G = np.asarray(dY, np.float64)
        for l in reversed(range(L)):
            A, Z = saved[l]
            dZ = timed("r", lambda: G * ((Z > 0) if l < L - 1 else 1.0))
            timed("r", orc.gemm, A.T, dZ, True)
            if l == 0:
                break
            dA = timed("r", orc.gemm, dZ, Ws[l].T, True).astype(np.float32)
            d = dA.shape[1]
            pk = timed("q", orc.quantize, dA, self.mask, bits, sb[l]) if bits < 32 else None
            M = timed("r", orc.messages, dA, pk, self.mask, d, bits)
            G = timed("e", orc.spmm, self.rp, self.col, orc.COEF_GCN, M, transpose=True)
        wall = time.perf_counter() - t_all
        self.last = {k: (t[k], scale[k]) for k in t}
        return sum(t[k] * scale[k] for k in t), wall

    def text(self, bits):
        return (f"row subset scaled linearly: {self.n_rows} seeded destination rows with their {self.e} in-edges "
                f"and the {self.nn} nodes they touch, the {len(self.w.widths) - 1}-layer stack "
                f"{' -> '.join(map(str, self.w.widths))} forward+backward at b = {bits}, float64 oracle; each "
                f"stage's time scaled by its units on the whole graph ({self.e_full} edges, {self.n_full} rows, "
                f"{self.m_full} quantized rows)")


def run_reference(args, w):
    """The oracle as it stands, on the host cores, on a bounded sample of the
    workload (the row subset above) at every step."""
    import oracle
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    g = w.make_graph(device=dev)
    mask = synth.bernoulli_mask(g.n, w.mask_frac, seed=w.seed, device=dev)
    smp = OracleSample(w, g, mask)
    X, Ws, dY = smp.inputs(synth.normal_matrix(g.n, w.widths[0], seed=w.seed, device=dev),
                           synth.normal_matrix(g.n, w.widths[-1], seed=w.seed, tag=synth.TAG_GRAD, device=dev))
    b = w.bits[0]
    for _ in range(args.warmup):
        smp.step(oracle, X, Ws, dY, b, w.seed)
    est, wall = [], []
    for _ in range(args.steps):
        e_, w_ = smp.step(oracle, X, Ws, dY, b, w.seed)
        est.append(e_)
        wall.append(w_)
    L = len(w.widths) - 1
    value = L * g.nnz / statistics.median(est)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sum(wall) / len(wall) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": gcn_config(w, g, 1),
            "scaled_step_s": statistics.median(est),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": smp.text(b)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(w, g, mask, X_full, dY_full, repeats=4):
    """Time the oracle on the bounded sample of the same workload."""
    import oracle
    oracle.build()
    smp = OracleSample(w, g, mask)
    X, Ws, dY = smp.inputs(X_full, dY_full)
    b = w.bits[0]
    est, wall = [], 0.0
    for _ in range(repeats):
        e_, w_ = smp.step(oracle, X, Ws, dY, b, w.seed)
        est.append(e_)
        wall += w_
    L = len(w.widths) - 1
    return {"value": L * g.nnz / statistics.median(est), "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle", "sample": smp.text(b) + f"; median of {repeats} sampled steps, {wall:.1f} s of CPU work"}


def gcn_config(w, g, ws):
    return {"workload": w.name, "nodes": g.n, "edges": g.nnz, "widths": list(w.widths),
            "bits": list(w.bits), "marginal_fraction": w.mask_frac, "coefficients": "gcn",
            "l2": "inputs larger than L2; also flushed (256 MiB write) before every timed step",
            "parallelism": "replicas" if ws > 1 else "single"}


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
        # the transposed aggregation of layer l > 0 writes layer l-1's dZ:
        # bf16, through the ReLU gate of layer l-1's output
        fused = not fwd and model.fuse_dz and l > 0
        c, s_ = spmm_bytes(g.n, g.nnz, d, b, n_marg, marg_out if fwd else marg_in, 2 if fwd or fused else 4, q,
                           gated=fused)
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
    roofline = {"kernel": "spmm_warp_kernel (de-quantizing aggregation, forward and transposed)",
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
            "config": gcn_config(w, g, ws),
            "roofline": roofline,
            "stage_ms_per_step": {k: round(v, 4) for k, v in stage_summary.items()},
            "e2e": e2e, "gpu_launches": launches}
    cs = clocks.summary()
    if cs is not None:
        line["clocks"] = cs
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, g, mask, X, dY)
    del model, G
    if rank == 0 and not args.no_largest and w.name == GCN3_LARGE.name:
        torch.cuda.empty_cache()
        line["roofline_largest"] = largest_aggregation(args, dev, q, flush)
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


def largest_aggregation(args, dev, q, flush, d=256, bits=8):
    """The de-quantizing aggregation alone on the largest graph (R-MAT,
    2^24 nodes, 32 draws per node, every row packed at `bits`, GCN
    coefficients), forward and transposed, each timed with CUDA events over
    args.steps launches after one untimed call (inputs larger than L2, L2
    also flushed before every launch)."""
    w = AGG_SWEEP
    t0 = time.perf_counter()
    g = w.make_graph(device=dev)
    G = q.graph_prepare(g.rowptr, g.col)
    X = synth.normal_matrix(g.n, d, seed=w.seed, device=dev)
    pk = q.quantize_pack(X, None, bits, 7)
    Y = torch.empty(g.n, d, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    t_setup = time.perf_counter() - t0
    n, E = g.n, g.nnz
    with ClockSampler(dev.index or 0) as clocks:
        torch.cuda.profiler.start()
        tf = _timed(lambda: q.dequant_spmm(G, None, pk, None, d, bits, out=Y), args.steps, flush)
        tb = _timed(lambda: q.dequant_spmm(G, None, pk, None, d, bits, transpose=True, out=Y), args.steps, flush)
        torch.cuda.profiler.stop()
    if int(G.status.cpu()[0]) != 0:
        raise RuntimeError(f"aggregation status word {int(G.status.cpu()[0]):#x}")
    pitch = q.packed_pitch(d, bits)
    comp = (n + 1) * 4 + E * 4 + 2 * n * 4 + n * pitch + n * d * 4
    stream = (n + 1) * 4 + E * 8 + n * 4 + E * pitch + n * d * 4
    peaks, kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    ms = (tf + tb) / 2
    achieved = comp / (ms / 1e3) / 1e9
    rec = {"workload": w.name, "nodes": n, "edges": E, "d": d, "bits": bits, "coefficients": "gcn",
           "kernel": "spmm_async_kernel (de-quantizing aggregation, every row packed)",
           "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
           "peak_source": f"hbm_gbs of {kind}", "traffic": load_traffic(f"{w.name}/d{d}b{bits}"),
           "algorithmic_bytes_per_launch": comp, "streaming_bytes_per_launch": stream,
           "fwd_ms": tf, "bwd_ms": tb, "launches_timed": 2 * args.steps,
           "edges_per_s": E / (ms / 1e3), "setup_s": t_setup,
           "l2": "inputs larger than L2; also flushed before every launch"}
    cs = clocks.summary()
    if cs is not None:
        rec["clocks"] = cs
    del G, X, pk, Y, g
    torch.cuda.empty_cache()
    return rec


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


def gemm_rates(args):
    """The dense int8 and bf16 GEMM rates of this GPU through cuBLAS
    (torch._int_mm with int32 accumulation, torch.matmul in bf16) on square
    shapes and on the update GEMM's shape of the large GCN workload: the
    measurement behind keeping the update GEMMs in bf16 (Tango Sec. 3.3 /
    4.3 take int8 GEMMs where int8 runs faster than fp16)."""
    dev = torch.device("cuda", 0)

    def timed(fn, iters=20):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(iters):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / iters

    out = {"measurement": "dense GEMM rates through cuBLAS", "unit": "TFLOP/s (int8: TOPS)"}
    shapes = [(n, n, n) for n in (4096, 8192)] + [(GCN3_LARGE.graph["n"], 256, 256)]
    for M, K, N in shapes:
        key = f"{M}x{K}x{N}"
        A = torch.randn(M, K, device=dev, dtype=torch.bfloat16)
        B = torch.randn(K, N, device=dev, dtype=torch.bfloat16)
        t = timed(lambda: A @ B)
        out[f"bf16_{key}"] = {"ms": t, "rate": 2 * M * K * N / t / 1e9}
        Ai = torch.randint(-100, 100, (M, K), device=dev, dtype=torch.int8)
        Bi = torch.randint(-100, 100, (K, N), device=dev, dtype=torch.int8)
        t = timed(lambda: torch._int_mm(Ai, Bi))
        out[f"int8_{key}"] = {"ms": t, "rate": 2 * M * K * N / t / 1e9}
        del A, B, Ai, Bi
    print(json.dumps(out), flush=True)


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
    ap.add_argument("--workload", default=GCN3_LARGE.name, choices=list(BY_NAME))
    ap.add_argument("--sweep-d", default=None, help="aggregate workload: comma-separated widths")
    ap.add_argument("--sweep-bits", default=None, help="aggregate workload: comma-separated bit-widths")
    ap.add_argument("--graph-scale", type=int, default=None,
                    help="aggregate / GAT workloads: R-MAT scale S (2^S nodes; 32 / 16 draws per node) for smaller cases")
    ap.add_argument("--alpha-bits", type=int, default=32, choices=[32, 8],
                    help="GAT workload: 8 quantizes the attention values the SpMM reads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-largest", action="store_true",
                    help="skip the record of the aggregation on the largest graph")
    ap.add_argument("--gemm-rates", action="store_true",
                    help="print the dense int8 and bf16 GEMM rates (cuBLAS) instead of a benchmark line")
    args = ap.parse_args()
    if args.gemm_rates:
        gemm_rates(args)
        return
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
