"""A graph without edges (rowptr all zero, an empty col), the degenerate case
of every edge kernel: the aggregations give zero rows, the edge softmax has
nothing to score, the attention-value headers are {0, 0}, and the GAT layer's
outputs and gradients are exactly zero (every sum over an empty edge set is
exactly 0, and so is every product with it)."""
import pytest
import torch

import synth
from gpu_helpers import gq

pytestmark = pytest.mark.gpu


def _edgeless(n=300):
    q = gq()
    rowptr = torch.zeros(n + 1, dtype=torch.int32, device="cuda")
    col = torch.zeros(0, dtype=torch.int32, device="cuda")
    return q, q.graph_prepare(rowptr, col)


@pytest.mark.parametrize("bits", [32, 4])
def test_aggregations_are_zero(bits):
    q, G = _edgeless()
    d, heads = 64, 4
    X = synth.normal_matrix(G.n, d, seed=1, device="cuda")
    pk = q.quantize_pack(X, None, bits, 3) if bits < 32 else None
    for transpose in (False, True):
        Y = q.dequant_spmm(G, X, pk, None, d, bits, coef=q.COEF_GCN, transpose=transpose)
        assert torch.count_nonzero(Y).item() == 0
        alpha = torch.zeros(0, heads, device="cuda")
        Y = q.edge_spmm(G, alpha, X, pk, None, d, bits, transpose=transpose)
        assert torch.count_nonzero(Y).item() == 0
    assert int(G.status.cpu()[0]) == 0


def test_softmax_and_attention_codes():
    q, G = _edgeless()
    heads = 4
    S = synth.normal_matrix(G.n, heads, seed=2, device="cuda")
    D = synth.normal_matrix(G.n, heads, seed=3, device="cuda")
    alpha = q.sddmm_edge_softmax(G, S, D)
    assert alpha.shape == (0, heads)
    codes, hdr = q.quantize_edge_values(G, alpha, 5)
    assert codes.shape == (0, heads) and torch.count_nonzero(hdr).item() == 0
    assert q.dequant_edge_values(G, codes, hdr).shape == (0, heads)
    X = synth.normal_matrix(G.n, 64, seed=4, device="cuda")
    assert torch.count_nonzero(q.edge_spmm_alpha8(G, codes, hdr, X, None, None, 64)).item() == 0
    assert int(G.status.cpu()[0]) == 0


@pytest.mark.parametrize("bits,alpha_bits", [(32, 32), (8, 8)])
def test_gat_layer_is_zero(bits, alpha_bits):
    q, G = _edgeless()
    d_in, heads, f = 32, 4, 16
    d = heads * f
    H = synth.normal_matrix(G.n, d_in, seed=5, device="cuda")
    W = synth.glorot(d_in, d, seed=6, device="cuda")
    a_s = synth.glorot(heads, f, seed=7, device="cuda")
    a_d = synth.glorot(heads, f, seed=8, device="cuda")
    mask = torch.ones(G.n, dtype=torch.uint8, device="cuda") if bits < 32 else None
    L = q.GATLayer(G, d_in, heads, f, 0.2, bits, mask, alpha_bits=alpha_bits)
    out = L.forward(H, W, a_s, a_d, 9)
    dOut = synth.normal_matrix(G.n, d, seed=10, tag=synth.TAG_GRAD, device="cuda")
    dW, das, dad, dH = L.backward(dOut, H, W, a_s, a_d, 11)
    torch.cuda.synchronize()
    assert int(L.err.item()) == 0 and int(G.status.cpu()[0]) == 0
    for t in (out, dW, das, dad, dH):
        assert torch.count_nonzero(t).item() == 0
    # the forward still ran its GEMM: H' = H W is not zero
    assert torch.count_nonzero(L.Hp).item() > 0
