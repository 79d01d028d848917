"""Shared helpers of the GPU parity tests (no method arithmetic here)."""
import numpy as np
import pytest
import torch

import synth


def require_cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def gq():
    require_cuda()
    import quantized_gnn_message_gb300 as q
    q.lib()
    return q


def close(gpu, ref, rtol=1e-4, what=""):
    """max |gpu - ref| <= rtol * (1 + |ref|), elementwise."""
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    err = np.abs(g - r) - rtol * (1.0 + np.abs(r))
    if err.size and err.max() > 0:
        i = np.unravel_index(np.argmax(err), err.shape)
        raise AssertionError(f"{what}: mismatch at {i}: gpu={g[i]!r} ref={r[i]!r} "
                             f"({int((err > 0).sum())} of {err.size} elements out of tolerance)")


def rmat_small(scale=12, n=3000, deg=12, seed=1):
    return synth.rmat_graph(scale=scale, n=n, n_draws=n * deg, seed=seed)


def hub_graph(n=3000, seed=3):
    """A graph with a dozen rows (in and out) above 256 edges, a heavier
    head up to ~650 edges, and a ragged tail of rows with few edges."""
    return synth.rmat_graph(scale=12, n=n, n_draws=n * 30, a=0.75, b=0.1, c=0.1, seed=seed)


def sparse_rows_graph(n=6000, seed=5):
    """CSR with rows of no edges (also first and last), many single-edge
    rows (runs of more than 32 rows), mid-size rows, a few hubs of 300-700
    edges and one of 2000 edges."""
    rng = np.random.default_rng(seed)
    kind = rng.random(n)
    deg = np.where(kind < 0.3, 0, np.where(kind < 0.7, 1, rng.integers(2, 40, n)))
    deg[rng.choice(n, 6, replace=False)] = rng.integers(300, 700, 6)
    deg[n // 2] = 2000          # a hub cut into several tasks
    deg[:3] = 0                 # rows without edges at both ends
    deg[-3:] = 0
    rowptr = np.zeros(n + 1, np.int64)
    rowptr[1:] = np.cumsum(deg)
    col = np.concatenate([np.sort(rng.choice(n, k, replace=False)) for k in deg]).astype(np.int32)
    return synth.Graph(n, torch.from_numpy(rowptr.astype(np.int32)), torch.from_numpy(col))


def sample_rows(rowptr, k, seed, n_heavy=None):
    """k destination rows: the heaviest rows (k // 4 unless given) plus a
    seeded uniform draw."""
    deg = np.diff(rowptr)
    heavy = np.argsort(-deg, kind="stable")[: k // 4 if n_heavy is None else n_heavy]
    rng = np.random.default_rng(seed)
    rest = rng.choice(deg.size, size=k - heavy.size, replace=False)
    return np.unique(np.concatenate([heavy, rest]))


def sub_csr(rowptr, col, rows):
    """The in-edges of `rows` as their own CSR (rows renumbered 0..m-1),
    their CSR edge ids, and their sources renumbered into `src` (the
    distinct sources, in ascending order)."""
    starts, ends = rowptr[rows], rowptr[rows + 1]
    eids = np.concatenate([np.arange(a, b) for a, b in zip(starts, ends)]).astype(np.int64)
    sub_rp = np.concatenate([[0], np.cumsum(ends - starts)]).astype(np.int32)
    src, local = np.unique(col[eids], return_inverse=True)
    return sub_rp, local.astype(np.int32), eids, src
