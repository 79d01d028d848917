"""Parity at the benchmark's full sizes, in the launch configurations
`bench.py` times.
  - The 3-layer GCN workload's graph (131,072 nodes, 2.75M edges, 40%
    marginal, d = 256): quantized bytes bit-exact and the de-quantizing
    aggregation, forward and transposed, on every row within 1e-4 (1 + |ref|)
    (the oracle finishes this size in seconds).
  - The GAT workload (1,048,576 nodes, 17.8M edges, 256 -> 4 x 64): on a
    sample of destination rows (the heaviest ones and a seeded draw), alpha,
    the layer's output and the backward's dE_pre within 1e-4, each row from
    its own in-edges (a row depends on nothing else), on the GPU's S, D and
    H'."""
import numpy as np
import pytest
import torch

import synth
from synth.configs import GAT_RMAT20, GCN3_RMAT17
from gpu_helpers import close, gq, sample_rows, sub_csr

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bits", [2, 8])
def test_headline_aggregation_full_size(orc, bits):
    q = gq()
    w = GCN3_RMAT17
    g = w.make_graph(device="cuda")
    G = q.graph_prepare(g.rowptr, g.col)
    rp, co = g.rowptr.cpu().numpy(), g.col.cpu().numpy()
    d = 256
    X = synth.normal_matrix(g.n, d, seed=w.seed + 11, device="cuda")
    mask = synth.bernoulli_mask(g.n, w.mask_frac, seed=w.seed, device="cuda")
    pk = q.quantize_pack(X, mask, bits, 12345)
    Xh, pkh, mh = X.cpu().numpy(), pk.cpu().numpy(), mask.cpu().numpy()
    sel = mh == 1
    np.testing.assert_array_equal(pkh[sel], orc.quantize(Xh, mh, bits, 12345)[sel])
    M = orc.messages(Xh, pkh, mh, d, bits)
    for transpose in (False, True):
        Y = q.dequant_spmm(G, X, pk, mask, d, bits, coef=q.COEF_GCN, transpose=transpose).cpu().numpy()
        close(Y, orc.spmm(rp, co, orc.COEF_GCN, M, transpose=transpose), what=f"b={bits} transpose={transpose}")
    assert int(G.status.cpu()[0]) == 0


def test_gat_full_size_sampled(orc):
    q = gq()
    w = GAT_RMAT20
    g = w.make_graph(device="cuda")
    G = q.graph_prepare(g.rowptr, g.col)
    d_in, heads, f = w.widths
    d = heads * f
    H = synth.normal_matrix(g.n, d_in, seed=w.seed, device="cuda")
    Wt = synth.glorot(d_in, d, seed=w.seed + 1, device="cuda")
    a_s = synth.glorot(heads, f, seed=w.seed + 2, device="cuda")
    a_d = synth.glorot(heads, f, seed=w.seed + 3, device="cuda")
    dOut = synth.normal_matrix(g.n, d, seed=w.seed, tag=synth.TAG_GRAD, device="cuda")
    L = q.GATLayer(G, d_in, heads, f, 0.2, 32, None)
    out = L.forward(H, Wt, a_s, a_d, 1)
    dEpre = torch.empty(g.nnz, heads, device="cuda")
    L.backward(dOut, H, Wt, a_s, a_d, 2, dEpre=dEpre)
    torch.cuda.synchronize()
    assert int(L.err.item()) == 0 and int(G.status.cpu()[0]) == 0

    rp, co = g.rowptr.cpu().numpy(), g.col.cpu().numpy()
    rows = sample_rows(rp, 160, seed=5, n_heavy=8)
    srp, scol, eids, src = sub_csr(rp, co, rows)
    idx = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    S = L.S[idx(src)].cpu().numpy()
    Dv = L.D[idx(rows)].cpu().numpy()
    Hp = L.Hp[idx(src)].cpu().numpy()
    ag = L.alpha[idx(eids)].cpu().numpy()
    Es, a_ref = orc.edge_softmax(srp, scol, S, Dv, 0.2)
    close(ag, a_ref, what="alpha")
    close(out[idx(rows)].cpu().numpy(), orc.edge_spmm(srp, scol, ag, Hp), what="out")
    da = orc.sddmm_dot(srp, scol, dOut[idx(rows)].cpu().numpy(), Hp, heads)
    _, _, dE_ref = orc.edge_softmax_bwd(srp, ag, da, Es, 0.2)
    close(dEpre[idx(eids)].cpu().numpy(), dE_ref, what="dE_pre")
