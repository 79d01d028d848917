"""Graph preparation on the GPU: CSR validation, degree norms bit-exact with
the oracle's (float)(1/sqrt((double)deg)), stable transpose, hub lists."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import gq, hub_graph

pytestmark = pytest.mark.gpu


def _check_sched(tasks, groups, ptr, thr, split, light=None):
    """Tasks cover exactly the edges of the rows heavier than thr, in pieces
    of at most `split` edges, heaviest rows first; split rows form groups."""
    deg = np.diff(ptr)
    heavy = np.nonzero(deg > thr)[0]
    cover = {}
    for t, (r, b, e, grp) in enumerate(tasks):
        assert deg[r] > thr and ptr[r] <= b < e <= ptr[r + 1] and e - b <= split
        cover.setdefault(r, []).append((b, e, grp, t))
    assert sorted(cover) == sorted(heavy.tolist())
    for r, pieces in cover.items():
        pieces.sort()
        assert pieces[0][0] == ptr[r] and pieces[-1][1] == ptr[r + 1]
        assert all(pieces[i][1] == pieces[i + 1][0] for i in range(len(pieces) - 1))
        if len(pieces) == 1:
            assert pieces[0][2] == -1
        else:
            gi = pieces[0][2]
            assert all(p[2] == gi for p in pieces)
            gr, first, cnt, _ = groups[gi]
            assert gr == r and cnt == len(pieces) and [p[3] for p in pieces] == list(range(first, first + cnt))
    first_task_deg = [deg[cover_r] for cover_r in [t[0] for t in tasks]]
    # light runs: consecutive light rows, every light row exactly once,
    # at most 256 edges per run unless the run is a single row
    if light is not None:
        seen = np.zeros(len(ptr) - 1, np.int32)
        for rb, re in light:
            assert rb < re and np.all(deg[rb:re] <= thr)
            assert ptr[re] - ptr[rb] <= 256 or re - rb == 1
            seen[rb:re] += 1
        np.testing.assert_array_equal(seen, (deg <= thr).astype(np.int32))
    assert all(first_task_deg[i] >= first_task_deg[i + 1] for i in range(len(first_task_deg) - 1))
    slots = [gr[3] for gr in groups]
    assert slots == list(np.cumsum([0] + [gr[2] for gr in groups])[:-1])


def _check(orc, g, hub_threshold=0, split_edges=0):
    q = gq()
    rp, co = g.rowptr.cuda(), g.col.cuda()
    G = q.graph_prepare(rp, co, hub_threshold, split_edges)
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
    thr, split = G.c.hub_threshold, G.c.split_edges
    for tr, ptr in ((False, rowptr), (True, np.concatenate([[0], np.cumsum(cnt)]))):
        tasks, groups = (x.cpu().numpy() for x in G.sched_arrays(tr))
        sc = G.c.tr_sched if tr else G.c.sched
        off = sc.light - G.storage.data_ptr()
        light = G.storage[off:off + sc.n_light * 8].view(torch.int32).view(-1, 2).cpu().numpy()
        _check_sched(tasks, groups, ptr, thr, split, light)
    assert G.c.max_deg == np.diff(rowptr).max() and G.c.tr_max_deg == cnt.max()
    return G


def test_prepare_uniform(orc):
    _check(orc, synth.uniform_graph(1024, 16384, seed=0))


def test_prepare_rmat_hubs(orc):
    G = _check(orc, hub_graph(), hub_threshold=64)
    assert G.n_tasks > 0 and G.tr_n_tasks > 0
    G = _check(orc, hub_graph(), hub_threshold=32, split_edges=256)
    assert G.c.sched.n_groups > 0 and G.c.tr_sched.n_groups > 0


def test_prepare_rejects_bad_schedule_args():
    q = gq()
    g = synth.uniform_graph(64, 256, seed=1)
    with pytest.raises(q.GQError, match="invalid"):
        q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), 16, 0)
    with pytest.raises(q.GQError, match="invalid"):
        q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), 64, 100)


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
