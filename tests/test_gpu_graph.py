"""Graph preparation on the GPU: CSR validation, degree norms bit-exact with
the oracle's (float)(1/sqrt((double)deg)), stable transpose, hub lists."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import gq, rmat_small, hub_graph

pytestmark = pytest.mark.gpu


def _check(orc, g, hub_threshold=0):
    q = gq()
    rp, co = g.rowptr.cuda(), g.col.cuda()
    G = q.graph_prepare(rp, co, hub_threshold)
    rowptr, col = g.rowptr.numpy(), g.col.numpy()
    n, nnz = g.n, g.nnz
    di, do, ii = orc.degree_norms(rowptr, col)
    np.testing.assert_array_equal(G.dinv_in.cpu().numpy(), di)
    np.testing.assert_array_equal(G.dinv_out.cpu().numpy(), do)
    np.testing.assert_array_equal(G.inv_in.cpu().numpy(), ii)
    # stable transpose: sort CSR entries by source, ties in CSR order
    perm = np.argsort(col, kind="stable")
    dst = np.repeat(np.arange(n), np.diff(rowptr))
    cnt = np.bincount(col, minlength=n)
    np.testing.assert_array_equal(G.tr_rowptr.cpu().numpy(), np.concatenate([[0], np.cumsum(cnt)]))
    np.testing.assert_array_equal(G.tr_perm.cpu().numpy(), perm)
    np.testing.assert_array_equal(G.tr_col.cpu().numpy(), dst[perm])
    thr = G.c.hub_threshold
    assert G.n_hub == int((np.diff(rowptr) > thr).sum())
    assert G.tr_n_hub == int((cnt > thr).sum())
    assert G.c.max_deg == np.diff(rowptr).max() and G.c.tr_max_deg == cnt.max()
    return G


def test_prepare_uniform(orc):
    _check(orc, synth.uniform_graph(1024, 16384, seed=0))


def test_prepare_rmat_hubs(orc):
    G = _check(orc, hub_graph(), hub_threshold=64)
    assert G.n_hub > 0 and G.tr_n_hub > 0


def test_prepare_rmat_medium(orc):
    # > 2^16 nodes: three radix passes, multi-level scans
    _check(orc, synth.rmat_graph(scale=17, n=100_000, n_draws=800_000, seed=4))


def test_prepare_single_node(orc):
    g = synth.Graph(1, torch.tensor([0, 1], dtype=torch.int32), torch.tensor([0], dtype=torch.int32))
    _check(orc, g)


def test_prepare_rejects_bad_graphs():
    q = gq()
    rp = torch.tensor([0, 2, 1, 3], dtype=torch.int32, device="cuda")   # decreasing
    co = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    with pytest.raises(q.GQError, match="validation"):
        q.graph_prepare(rp, co)
    rp = torch.tensor([0, 1, 2, 3], dtype=torch.int32, device="cuda")
    co = torch.tensor([0, 5, 2], dtype=torch.int32, device="cuda")      # col out of range
    with pytest.raises(q.GQError, match="validation"):
        q.graph_prepare(rp, co)
    co = torch.tensor([0, -1, 2], dtype=torch.int32, device="cuda")
    with pytest.raises(q.GQError, match="validation"):
        q.graph_prepare(rp, co)
    rp = torch.tensor([0, 1, 2, 4], dtype=torch.int32, device="cuda")   # rowptr[n] != nnz
    with pytest.raises(q.GQError, match="validation"):
        q.graph_prepare(rp, co)
