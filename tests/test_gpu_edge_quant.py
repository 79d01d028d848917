"""8-bit attention values on the GPU vs the oracle (Tango Sec. 3.3: the
SpMM reads quantized edge features; each (destination, head) segment is one
AdaQP Eqn 4 vector): codes and {S, Z} headers bit-exact on the same fp32
input, de-quantized values bit-exact, and the multi-head SpMM over the codes
within 1e-4 (1 + |ref|) of the oracle's SpMM of the de-quantized values."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import close, gq, hub_graph, rmat_small, sparse_rows_graph

pytestmark = pytest.mark.gpu

GRAPHS = ["uniform", "rmat", "hubs_split", "sparse_rows"]


def _graph(q, name):
    if name == "uniform":
        g, kw = synth.uniform_graph(1024, 16384, seed=0), {}
    elif name == "rmat":
        g, kw = rmat_small(), {}
    elif name == "sparse_rows":  # rows without edges, 1-edge rows, 2-39-edge rows, hubs
        g, kw = sparse_rows_graph(), dict(hub_threshold=600, split_edges=512)
    else:  # heavy rows split into several tasks
        g, kw = hub_graph(), dict(hub_threshold=32, split_edges=256)
    return g, q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), **kw)


def _alpha(q, g, G, heads, kind):
    if kind == "softmax":
        S = synth.normal_matrix(g.n, heads, seed=heads) * 2
        D = synth.normal_matrix(g.n, heads, seed=heads + 9) * 2
        return q.sddmm_edge_softmax(G, S.cuda(), D.cuda(), slope=0.2)
    # arbitrary finite values, negative ones included
    return synth.normal_matrix(g.nnz, heads, seed=heads + 3, device="cuda")


@pytest.mark.parametrize("graph", GRAPHS)
@pytest.mark.parametrize("heads", [1, 2, 4, 8])
@pytest.mark.parametrize("kind", ["softmax", "normal"])
def test_codes_and_headers_bit_exact(orc, graph, heads, kind):
    q = gq()
    g, G = _graph(q, graph)
    if graph == "hubs_split":
        assert G.c.sched.n_groups > 0
    alpha = _alpha(q, g, G, heads, kind)
    torch.cuda.synchronize()  # the softmax's own errors surface here
    codes, hdr = q.quantize_edge_values(G, alpha, 77)
    torch.cuda.synchronize()
    a = alpha.cpu().numpy()
    rp = g.rowptr.numpy()
    c_ref, h_ref = orc.quantize_edge_values(rp, a, 77)
    np.testing.assert_array_equal(codes.cpu().numpy(), c_ref)
    np.testing.assert_array_equal(hdr.cpu().numpy(), h_ref)
    deq = q.dequant_edge_values(G, codes, hdr).cpu().numpy()
    np.testing.assert_array_equal(deq, orc.dequant_edge_values(rp, c_ref, h_ref))
    assert int(G.status.cpu()[0]) == 0


@pytest.mark.parametrize("graph", GRAPHS)
@pytest.mark.parametrize("heads,f", [(1, 16), (2, 32), (4, 16), (4, 64), (8, 32)])
@pytest.mark.parametrize("bits", [32, 4])
def test_spmm_over_codes(orc, graph, heads, f, bits):
    q = gq()
    g, G = _graph(q, graph)
    d = heads * f
    alpha = _alpha(q, g, G, heads, "softmax")
    codes, hdr = q.quantize_edge_values(G, alpha, 5)
    X = synth.normal_matrix(g.n, d, seed=d + bits)
    mask = synth.bernoulli_mask(g.n, 0.5, seed=2)
    Xd = X.cuda()
    md = mask.cuda() if bits < 32 else None
    pk = q.quantize_pack(Xd, md, bits, 9) if bits < 32 else None
    Y = q.edge_spmm_alpha8(G, codes, hdr, Xd, pk, md, d, bits).cpu().numpy()
    rp, co = g.rowptr.numpy(), g.col.numpy()
    ahat = orc.dequant_edge_values(rp, codes.cpu().numpy(), hdr.cpu().numpy())
    M = orc.messages(X.numpy(), None if pk is None else pk.cpu().numpy(), mask.numpy(), d, bits)
    close(Y, orc.edge_spmm(rp, co, ahat, M), what=f"{graph} heads={heads} f={f} bits={bits}")
    assert int(G.status.cpu()[0]) == 0


def test_empty_graph_rows_and_arguments():
    q = gq()
    g, G = _graph(q, "sparse_rows")
    alpha = _alpha(q, g, G, 4, "softmax")
    codes, hdr = q.quantize_edge_values(G, alpha, 1)
    h = hdr.cpu().numpy()
    empty = np.diff(g.rowptr.numpy()) == 0
    assert empty.any() and np.all(h[empty] == 0.0)
    X = synth.normal_matrix(g.n, 512, seed=1, device="cuda")
    with pytest.raises(q.GQError):  # d above 256
        q.edge_spmm_alpha8(G, codes, hdr, X, None, None, 512)
    X3 = synth.normal_matrix(g.n, 48, seed=1, device="cuda")
    with pytest.raises(q.GQError):  # head width 12 is not a power of two >= 16
        q.edge_spmm_alpha8(G, codes, hdr, X3, None, None, 48)
    a3 = torch.zeros(g.nnz, 3, device="cuda")
    with pytest.raises(q.GQError):  # heads = 3
        q.quantize_edge_values(G, a3, 1)
