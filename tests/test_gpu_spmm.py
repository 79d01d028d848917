"""Dequant-fused SpMM on the GPU vs the oracle (AdaQP Sec. 2.1/3.1, Eqn 5;
Sancus Sec. 2): forward and transposed, GCN / SAGE / plain coefficients,
2/4/8-bit and unquantized messages, mixed masks, power-law hubs (block
path) and a ragged tail.  The oracle aggregates the messages de-quantized
from the GPU's own packed bytes (per-stage check), in float64;
tolerance max|gpu - ref| <= 1e-4 (1 + |ref|)."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import gq, close, rmat_small, hub_graph, sparse_rows_graph

pytestmark = pytest.mark.gpu


def _spmm_case(orc, g, d, bits, coef, transpose, mask_frac, hub_threshold=0, seed=0, split_edges=0):
    q = gq()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), hub_threshold, split_edges)
    X = synth.normal_matrix(g.n, d, seed=seed + d).numpy()
    mask = None if mask_frac is None else synth.bernoulli_mask(g.n, mask_frac, seed=seed + 1).numpy()
    Xd = torch.from_numpy(X).cuda()
    md = None if mask is None else torch.from_numpy(mask).cuda()
    pk = None
    if bits < 32:
        pk = q.quantize_pack(Xd, md, bits, seed + 7)
    Y = q.dequant_spmm(G, Xd, pk, md, d, bits, coef=coef, transpose=transpose).cpu().numpy()
    M = orc.messages(X, None if pk is None else pk.cpu().numpy(), mask, d, bits)
    ref = orc.spmm(g.rowptr.numpy(), g.col.numpy(), coef, M, transpose=transpose)
    close(Y, ref, what=f"spmm d={d} bits={bits} coef={coef} T={transpose}")
    assert int(G.status.cpu()[0]) == 0  # no bounded wait gave up
    return G


@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("bits", [2, 4, 8, 32])
@pytest.mark.parametrize("coef", [0, 1, 2])
def test_spmm_uniform(orc, transpose, bits, coef):
    g = synth.uniform_graph(1024, 16384, seed=0)
    _spmm_case(orc, g, 64, bits, coef, transpose, 0.3)


@pytest.mark.parametrize("d", [4, 12, 32, 64, 100, 128, 256, 384, 1024])
@pytest.mark.parametrize("bits", [2, 8, 32])
def test_spmm_widths(orc, d, bits):
    _spmm_case(orc, rmat_small(), d, bits, 0, False, 0.5)
    _spmm_case(orc, rmat_small(), d, bits, 0, True, 0.5)


@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("bits", [4, 32])
@pytest.mark.parametrize("d", [32, 256, 512])
@pytest.mark.parametrize("split", [0, 256])
def test_spmm_heavy_rows(orc, transpose, bits, d, split):
    G = _spmm_case(orc, hub_graph(), d, bits, 0, transpose, 0.4, hub_threshold=48, split_edges=split)
    sc = G.c.tr_sched if transpose else G.c.sched
    assert sc.n_tasks > 0
    if split:
        assert sc.n_groups > 0


@pytest.mark.parametrize("bits", [2, 8])
def test_spmm_all_marginal_no_X(orc, bits):
    # mask == NULL: every message row is read from the packed buffer, X unused
    q = gq()
    g = rmat_small()
    d = 64
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda())
    X = synth.normal_matrix(g.n, d, seed=3).numpy()
    pk = q.quantize_pack(torch.from_numpy(X).cuda(), None, bits, 5)
    Y = q.dequant_spmm(G, None, pk, None, d, bits).cpu().numpy()
    ref = orc.spmm(g.rowptr.numpy(), g.col.numpy(), 0, orc.dequant(pk.cpu().numpy(), d, bits).astype(np.float64))
    close(Y, ref)


def test_spmm_deterministic(orc):
    q = gq()
    g = hub_graph()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), 32, 256)
    X = synth.normal_matrix(g.n, 128, seed=1, device="cuda")
    pk = q.quantize_pack(X, None, 4, 1)
    a = q.dequant_spmm(G, X, pk, None, 128, 4)
    b = q.dequant_spmm(G, X, pk, None, 128, 4)
    assert torch.equal(a, b)


@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("bits", [8, 32])
def test_edge_spmm(orc, transpose, bits):
    q = gq()
    g = hub_graph()
    heads, F = 4, 16
    d = heads * F
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), 40, 256)
    alpha = np.random.default_rng(2).random((g.nnz, heads)).astype(np.float32)
    X = synth.normal_matrix(g.n, d, seed=2).numpy()
    mask = synth.bernoulli_mask(g.n, 0.5, seed=3).numpy()
    Xd, md = torch.from_numpy(X).cuda(), torch.from_numpy(mask).cuda()
    pk = q.quantize_pack(Xd, md, bits, 9) if bits < 32 else None
    Y = q.edge_spmm(G, torch.from_numpy(alpha).cuda(), Xd, pk, md, d, bits, transpose=transpose).cpu().numpy()
    M = orc.messages(X, None if pk is None else pk.cpu().numpy(), mask, d, bits)
    ref = orc.edge_spmm(g.rowptr.numpy(), g.col.numpy(), alpha, M, transpose=transpose)
    close(Y, ref)


@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("d", [68, 128, 196, 256])
def test_spmm_sparse_rows(orc, transpose, bits, d):
    _spmm_case(orc, sparse_rows_graph(), d, bits, 0, transpose, 0.45, hub_threshold=64, split_edges=256)
    _spmm_case(orc, sparse_rows_graph(), d, bits, 1, transpose, 0.45)
