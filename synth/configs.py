"""The five synthetic workloads: graph recipe, widths, marginal fraction and
bit-widths.  Graph sizes follow the published node/edge counts of the
datasets they stand in for (ogbn-products for the large GCN); the graphs
themselves are seeded R-MAT or uniform draws (see synth.rmat_graph)."""
from __future__ import annotations

from dataclasses import dataclass, field

import synth


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                      # "gcn", "gat" or "aggregate"
    graph: dict                    # keyword args of the graph generator
    widths: tuple                  # layer widths d_0 -> d_1 -> ... (gcn) / (d_in, heads, f) (gat)
    mask_frac: float               # fraction of nodes marked marginal
    bits: tuple                    # quantization bit-widths run (32 = none)
    seed: int = 0
    sweep_d: tuple = field(default=())

    def make_graph(self, device="cpu") -> synth.Graph:
        g = dict(self.graph)
        kind = g.pop("kind")
        if kind == "uniform":
            return synth.uniform_graph(device=device, seed=self.seed, **g)
        return synth.rmat_graph(device=device, seed=self.seed, **g)


TINY_GCN = Workload(
    name="tiny-gcn-uniform-1k",
    kind="gcn",
    graph=dict(kind="uniform", n=1024, n_edges=16384),
    widths=(64, 64), mask_frac=0.30, bits=(8,))

GCN3_RMAT17 = Workload(
    name="gcn3-rmat17-131k",
    kind="gcn",
    graph=dict(kind="rmat", scale=17, n=131072, n_draws=20 * 131072,
               exact_edges=20 * 131072),
    widths=(128, 256, 256, 47), mask_frac=0.40, bits=(2, 4, 8))

GAT_RMAT20 = Workload(
    name="gat-rmat20-1m",
    kind="gat",
    graph=dict(kind="rmat", scale=20, n=1048576, n_draws=16 * 1048576,
               exact_edges=16 * 1048576),
    widths=(256, 4, 64), mask_frac=0.0, bits=(32,))

GCN3_LARGE = Workload(
    name="gcn3-rmat22-2.45m",
    kind="gcn",
    graph=dict(kind="rmat", scale=22, n=2449029, n_draws=61859140,
               exact_edges=61859140),
    widths=(100, 256, 256, 47), mask_frac=0.60, bits=(2,))

AGG_SWEEP = Workload(
    name="aggregate-rmat24-16.8m",
    kind="aggregate",
    graph=dict(kind="rmat", scale=24, n=16777216, n_draws=32 * 16777216),
    widths=(), mask_frac=1.0, bits=(2, 4, 8), sweep_d=(32, 64, 128, 256))

ALL = (TINY_GCN, GCN3_RMAT17, GAT_RMAT20, GCN3_LARGE, AGG_SWEEP)
BY_NAME = {w.name: w for w in ALL}
