"""GAT layer on the GPU vs the oracle (Tango Sec. 2.1, Fig. 1a/1b), stage by
stage on the GPU's own stage inputs:
  SDDMM add + LeakyReLU + edge softmax  alpha, E_pre        (1e-4)
  H' = H W                              bf16 GEMM           (2e-2 bar, 1e-3 check)
  S, D head projections of the GPU's H'                     (1e-4)
  out = multi-head SpMM of the GPU's alpha and messages     (1e-4)
  backward: dE_pre (SDDMM dot, softmax derivative, LeakyReLU'), dH' (dM +
  dS a_src + dD a_dst), da_src / da_dst, dW, dH."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import close, gq, hub_graph, rmat_small, sparse_rows_graph

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("heads", [1, 2, 4, 8])
@pytest.mark.parametrize("graph", ["uniform", "rmat", "hubs_split", "sparse_rows"])
def test_edge_softmax(orc, heads, graph):
    q = gq()
    if graph == "uniform":
        g, kw = synth.uniform_graph(1024, 16384, seed=0), {}
    elif graph == "rmat":
        g, kw = rmat_small(), {}
    elif graph == "sparse_rows":  # rows without edges, 1-edge rows, 2-39-edge rows, hubs
        g, kw = sparse_rows_graph(), dict(hub_threshold=600, split_edges=512)
    else:
        g, kw = hub_graph(), dict(hub_threshold=32, split_edges=256)
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), **kw)
    S = synth.normal_matrix(g.n, heads, seed=heads) * 2
    D = synth.normal_matrix(g.n, heads, seed=heads + 9) * 2
    alpha, Epre = q.sddmm_edge_softmax(G, S.cuda(), D.cuda(), slope=0.2, with_epre=True)
    E_ref, a_ref = orc.edge_softmax(g.rowptr.numpy(), g.col.numpy(), S.numpy(), D.numpy(), 0.2)
    close(Epre.cpu().numpy(), E_ref, what="E_pre")
    close(alpha.cpu().numpy(), a_ref, what="alpha")


def _gat(orc, g, d_in, heads, f, bits, mask_frac, kw, seed=0, alpha_bits=32):
    q = gq()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), **kw)
    rp, co = g.rowptr.numpy(), g.col.numpy()
    d = heads * f
    H = synth.normal_matrix(g.n, d_in, seed=seed + 1)
    W = synth.glorot(d_in, d, seed=seed + 2)
    a_s = synth.glorot(heads, f, seed=seed + 3)
    a_d = synth.glorot(heads, f, seed=seed + 4)
    mask = synth.bernoulli_mask(g.n, mask_frac, seed=seed + 5)
    dOut = synth.normal_matrix(g.n, d, seed=seed + 6, tag=synth.TAG_GRAD)
    sf, sb = synth.layer_seed(seed, 0, False), synth.layer_seed(seed, 0, True)
    L = q.GATLayer(G, d_in, heads, f, 0.2, bits, mask.cuda() if bits < 32 else None, alpha_bits=alpha_bits)
    Hd, Wd, asd, add_ = H.cuda(), W.cuda(), a_s.cuda(), a_d.cuda()
    out = L.forward(Hd, Wd, asd, add_, sf)
    dEpre = torch.empty(g.nnz, heads, device="cuda")
    dHp = torch.empty(g.n, d, device="cuda")
    dW, das, dad, dH = L.backward(dOut.cuda(), Hd, Wd, asd, add_, sb, dEpre=dEpre, dHp=dHp)
    torch.cuda.synchronize()
    assert int(L.err.item()) == 0

    Hp = L.Hp.cpu().numpy()
    Hp_ref = orc.gemm(H.numpy(), W.numpy(), bf16=True)
    close(Hp, Hp_ref, rtol=2e-2, what="H' bar")
    close(Hp, Hp_ref, rtol=1e-3, what="H'")
    close(L.S.cpu().numpy(), orc.head_proj(Hp, a_s.numpy(), heads), what="S")
    close(L.D.cpu().numpy(), orc.head_proj(Hp, a_d.numpy(), heads), what="D")
    Sg, Dg = L.S.cpu().numpy(), L.D.cpu().numpy()
    Epre_ref, a_ref = orc.edge_softmax(rp, co, Sg, Dg, 0.2)
    close(L.alpha.cpu().numpy(), a_ref, what="alpha")
    ag = L.alpha.cpu().numpy()
    mn = mask.numpy()
    pk = L.packed.cpu().numpy() if bits < 32 else None
    if bits < 32:
        ref_pk = orc.quantize(Hp, mn, bits, sf)
        np.testing.assert_array_equal(pk[mn == 1], ref_pk[mn == 1])
    M = orc.messages(Hp, pk, mn, d, bits)
    ahat = ag
    if alpha_bits == 8:  # the attention codes of the GPU's alpha, bit-exact
        c_ref, h_ref = orc.quantize_edge_values(rp, ag, sf ^ orc.ALPHA_SEED_TAG)
        np.testing.assert_array_equal(L.acode.cpu().numpy(), c_ref)
        np.testing.assert_array_equal(L.ahdr.cpu().numpy(), h_ref)
        ahat = orc.dequant_edge_values(rp, c_ref, h_ref)
    close(out.cpu().numpy(), orc.edge_spmm(rp, co, ahat, M), what="out")

    # backward, teacher-forced on the GPU's forward tensors
    dalpha = orc.sddmm_dot(rp, co, dOut.numpy(), M, heads)
    _, _, dEpre_ref = orc.edge_softmax_bwd(rp, ag, dalpha, Epre_ref, 0.2)
    close(dEpre.cpu().numpy(), dEpre_ref, what="dE_pre")
    dD_ref, dS_ref = orc.edge_segment_sums(rp, co, dEpre.cpu().numpy())
    dO = dOut.numpy()
    pkb = orc.quantize(dO, mn, bits, sb) if bits < 32 else None
    dM_ref = orc.edge_spmm(rp, co, ahat, orc.messages(dO, pkb, mn, d, bits), transpose=True)
    F = f
    dHp_ref = dM_ref + np.repeat(dS_ref, F, 1) * a_s.numpy().reshape(1, d) + np.repeat(dD_ref, F, 1) * a_d.numpy().reshape(1, d)
    close(dHp.cpu().numpy(), dHp_ref, what="dH'")
    close(das.cpu().numpy(), (dS_ref[:, :, None] * Hp.reshape(g.n, heads, F)).sum(0), rtol=1e-4, what="da_src")
    close(dad.cpu().numpy(), (dD_ref[:, :, None] * Hp.reshape(g.n, heads, F)).sum(0), rtol=1e-4, what="da_dst")
    dHg = dHp.cpu().numpy()
    dW_ref = orc.gemm(H.numpy().T, dHg, bf16=True)
    close(dW.cpu().numpy(), dW_ref, rtol=2e-2, what="dW bar")
    close(dW.cpu().numpy(), dW_ref, rtol=1e-3, what="dW")
    dH_ref = orc.gemm(dHg, W.numpy().T, bf16=True)
    close(dH.cpu().numpy(), dH_ref, rtol=1e-3, what="dH")


@pytest.mark.parametrize("heads,f", [(4, 64), (2, 32), (1, 16), (8, 32)])
def test_gat_layer(orc, heads, f):
    _gat(orc, rmat_small(), 256, heads, f, 32, 0.0, {})


@pytest.mark.parametrize("bits", [2, 8])
def test_gat_layer_quantized(orc, bits):
    _gat(orc, rmat_small(), 128, 4, 64, bits, 0.5, {})


def test_gat_layer_heavy_rows(orc):
    _gat(orc, hub_graph(), 100, 4, 32, 32, 0.0, dict(hub_threshold=32, split_edges=256))
    _gat(orc, hub_graph(), 64, 4, 16, 4, 0.4, dict(hub_threshold=32, split_edges=256))


@pytest.mark.parametrize("bits", [32, 4])
def test_gat_layer_quantized_alpha(orc, bits):
    _gat(orc, rmat_small(), 128, 4, 64, bits, 0.5, {}, alpha_bits=8)
    _gat(orc, hub_graph(), 64, 2, 32, bits, 0.4, dict(hub_threshold=32, split_edges=256), alpha_bits=8)
