"""Seeded synthetic inputs for the quantized message-passing layer.

This module is the only code shared by the CUDA path's tests/benchmarks and
the CPU oracle.  It holds no arithmetic of the method itself (no quantizer, no
coefficients, no aggregation): only deterministic generators of graphs,
feature matrices, weights, marginal masks and upstream gradients.

Every generator is a pure function of (seed, index) through a counter hash,
written with torch integer ops, so it yields the same bytes on the CPU and on
a GPU.  Floating-point outputs (Box-Muller normals, Glorot weights) are made
in float64 and rounded once to float32; callers that need identical bytes on
both sides generate once and copy.

The datasets the pages train on (Reddit, ogbn-products, AmazonProducts, ...)
are not available; these graphs stand in for them with matched node/edge
counts and a heavy-tailed (R-MAT) degree distribution.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

_M32 = 0xFFFFFFFF

# Stream tags: each generator draws from its own hash stream.
TAG_GRAPH = 0x47
TAG_FEAT = 0x46
TAG_WEIGHT = 0x57
TAG_MASK = 0x4D
TAG_GRAD = 0x44


def _mul32(h: torch.Tensor, c: int) -> torch.Tensor:
    """(h * c) mod 2**32 for int64 tensors holding uint32 values, without
    relying on int64 overflow behaviour."""
    lo = h * (c & 0xFFFF)
    hi = ((h * (c >> 16)) & 0xFFFF) << 16
    return (lo + hi) & _M32


def _fmix32(h: torch.Tensor) -> torch.Tensor:
    h = h ^ (h >> 16)
    h = _mul32(h, 0x85EBCA6B)
    h = h ^ (h >> 13)
    h = _mul32(h, 0xC2B2AE35)
    h = h ^ (h >> 16)
    return h


def hash_u32(seed: int, row: torch.Tensor, col) -> torch.Tensor:
    """32-bit counter hash of (seed, row, col); row/col int64 tensors (or an
    int for col).  Returns int64 tensor of uint32 values."""
    s32 = (seed & _M32) ^ ((seed >> 32) & _M32)
    dev = row.device
    ks = _fmix32(torch.tensor([s32], dtype=torch.int64, device=dev))
    kr = _fmix32((row & _M32) ^ ks)
    if not torch.is_tensor(col):
        col = torch.full_like(row, int(col))
    return _fmix32((kr + _mul32(col & _M32, 0x9E3779B9)) & _M32)


def uniform01(seed: int, row: torch.Tensor, col) -> torch.Tensor:
    """Float64 uniforms in [0, 1) with 32 random bits."""
    return hash_u32(seed, row, col).to(torch.float64) * (1.0 / 4294967296.0)


def stream_seed(base: int, tag: int) -> int:
    return (base ^ (tag << 40)) & 0xFFFFFFFFFFFFFFFF


# --------------------------------------------------------------------------
# graphs
# --------------------------------------------------------------------------

@dataclass
class Graph:
    """CSR by destination: row v lists the sources u of edges u->v (ascending),
    including exactly one self-loop per node.  int32 arrays."""
    n: int
    rowptr: torch.Tensor
    col: torch.Tensor

    @property
    def nnz(self) -> int:
        return int(self.col.numel())

    def to(self, device) -> "Graph":
        return Graph(self.n, self.rowptr.to(device), self.col.to(device))


def _csr_from_keys(n: int, keys: torch.Tensor) -> Graph:
    """keys = dst * n + src, unique, no self-loops.  Adds self-loops, sorts."""
    dev = keys.device
    loops = torch.arange(n, dtype=torch.int64, device=dev) * (n + 1)
    keys = torch.cat([keys, loops])
    keys, _ = torch.sort(keys)
    dst = keys // n
    src = keys - dst * n
    counts = torch.bincount(dst, minlength=n)
    rowptr = torch.zeros(n + 1, dtype=torch.int64, device=dev)
    rowptr[1:] = torch.cumsum(counts, 0)
    return Graph(n, rowptr.to(torch.int32), src.to(torch.int32))


def uniform_graph(n: int, n_edges: int, seed: int = 0, device="cpu") -> Graph:
    """Directed graph with `n_edges` distinct (src, dst) pairs, src != dst,
    endpoints uniform; the first `n_edges` distinct pairs in draw order."""
    gseed = stream_seed(seed, TAG_GRAPH)
    need = n_edges
    n_draw = int(n_edges * 1.3) + 64
    while True:
        i = torch.arange(n_draw, dtype=torch.int64, device=device)
        src = hash_u32(gseed, i, 0) % n
        dst = hash_u32(gseed, i, 1) % n
        keep = src != dst
        keys = (dst * n + src)[keep]
        order = i[keep]
        firsts = _first_occurrences(keys, order)
        if firsts.shape[1] >= need:
            break
        n_draw *= 2
    return _csr_from_keys(n, firsts[1, :need])


def _first_occurrences(keys: torch.Tensor, order: torch.Tensor):
    """Distinct keys in order of first appearance.  Returns a (2, m) tensor
    [draw index; key] sorted by draw index."""
    sk, perm = torch.sort(keys, stable=True)
    first = torch.ones_like(sk, dtype=torch.bool)
    first[1:] = sk[1:] != sk[:-1]
    fk = sk[first]
    fo = order[perm[first]]
    fo, p2 = torch.sort(fo)
    return torch.stack([fo, fk[p2]])


def rmat_graph(scale: int, n: int, n_draws: int, a=0.57, b=0.19, c=0.19,
               seed: int = 0, exact_edges: int | None = None, device="cpu",
               chunk: int = 1 << 26) -> Graph:
    """R-MAT graph: each draw descends `scale` levels of the 2^scale square
    adjacency matrix, choosing quadrant (src bit, dst bit) = (0,0) w.p. a,
    (0,1) w.p. b, (1,0) w.p. c, (1,1) otherwise.  Draws with an endpoint >= n
    and generator self-edges are dropped, duplicates removed.  With
    `exact_edges`, the first `exact_edges` distinct pairs in draw order are
    kept (more draws are made if needed)."""
    gseed = stream_seed(seed, TAG_GRAPH)
    ab, abc = a + b, a + b + c

    def draw(lo, hi):
        i = torch.arange(lo, hi, dtype=torch.int64, device=device)
        src = torch.zeros_like(i)
        dst = torch.zeros_like(i)
        for lvl in range(scale):
            u = uniform01(gseed, i, lvl)
            sb = (u >= ab).to(torch.int64)
            db = (((u >= a) & (u < ab)) | (u >= abc)).to(torch.int64)
            src = src * 2 + sb
            dst = dst * 2 + db
        keep = (src < n) & (dst < n) & (src != dst)
        return (dst * n + src)[keep], i[keep]

    if exact_edges is None:
        parts = []
        for lo in range(0, n_draws, chunk):
            k, _ = draw(lo, min(n_draws, lo + chunk))
            parts.append(torch.unique(k))
        keys = torch.unique(torch.cat(parts))
        return _csr_from_keys(n, keys)

    total = 0
    kparts, oparts = [], []
    nd = n_draws
    while True:
        for lo in range(total, nd, chunk):
            k, o = draw(lo, min(nd, lo + chunk))
            kparts.append(k)
            oparts.append(o)
        total = nd
        firsts = _first_occurrences(torch.cat(kparts), torch.cat(oparts))
        if firsts.shape[1] >= exact_edges:
            return _csr_from_keys(n, firsts[1, :exact_edges])
        nd = int(nd * 1.25) + 1024


# --------------------------------------------------------------------------
# dense inputs
# --------------------------------------------------------------------------

def normal_matrix(n: int, d: int, seed: int, tag: int = TAG_FEAT,
                  device="cpu", row0: int = 0) -> torch.Tensor:
    """n x d float32, entries ~ N(0,1) by Box-Muller from hash uniforms.
    Row r of the result is row (row0 + r) of the infinite stream."""
    s = stream_seed(seed, tag)
    out = torch.empty(n, d, dtype=torch.float32, device=device)
    step = max(1, (1 << 24) // max(d, 1))
    cols = torch.arange(d, dtype=torch.int64, device=device)
    for lo in range(0, n, step):
        hi = min(n, lo + step)
        r = torch.arange(row0 + lo, row0 + hi, dtype=torch.int64, device=device)
        rr = r[:, None].expand(hi - lo, d).reshape(-1)
        cc = cols[None, :].expand(hi - lo, d).reshape(-1)
        u1 = 1.0 - uniform01(s, rr, 2 * cc)
        u2 = uniform01(s, rr, 2 * cc + 1)
        z = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * math.pi * u2)
        out[lo:hi] = z.view(hi - lo, d).to(torch.float32)
    return out


def glorot(fan_in: int, fan_out: int, seed: int, tag: int = TAG_WEIGHT,
           device="cpu") -> torch.Tensor:
    """fan_in x fan_out float32, U(-r, r) with r = sqrt(6/(fan_in+fan_out))."""
    s = stream_seed(seed, tag)
    r = math.sqrt(6.0 / (fan_in + fan_out))
    i = torch.arange(fan_in * fan_out, dtype=torch.int64, device=device)
    u = uniform01(s, i // fan_out, i % fan_out)
    return ((2.0 * u - 1.0) * r).to(torch.float32).view(fan_in, fan_out)


def bernoulli_mask(n: int, frac: float, seed: int, tag: int = TAG_MASK,
                   device="cpu") -> torch.Tensor:
    """uint8 per node: 1 with probability `frac` (a 'marginal' node)."""
    s = stream_seed(seed, tag)
    i = torch.arange(n, dtype=torch.int64, device=device)
    return (uniform01(s, i, 0) < frac).to(torch.uint8)


def layer_seed(base: int, layer: int, backward: bool, which: int = 0) -> int:
    """Seed for the stochastic-rounding stream of one quantization site:
    base xor (tag << 32), tag = layer << 8 | direction << 4 | which."""
    tag = (layer << 8) | ((1 if backward else 0) << 4) | which
    return (base ^ (tag << 32)) & 0xFFFFFFFFFFFFFFFF
