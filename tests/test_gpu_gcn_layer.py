"""GCN / GraphSAGE-mean layer on the GPU vs the oracle, stage by stage on
the GPU's own stage inputs (AdaQP Sec. 2.1/3.1; Sancus Sec. 2):
  A      vs oracle aggregation of the same messages  (bf16 output: 5e-3)
  H_out  vs act(A_gpu W) in float64 on bf16 inputs   (2e-2 bar, 1e-3 check)
  dW, dA vs float64 products on bf16 inputs          (2e-2 bar, 1e-3 check)
  dH_in  vs oracle transposed aggregation of dA_gpu's messages (1e-4)
Quantized bytes of both passes are reproduced bit for bit by the oracle."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import gq, close, rmat_small, hub_graph

pytestmark = pytest.mark.gpu


def _case(orc, g, d_in, d_out, bits, act, coef, mask_frac=0.3, seed=0, hub_threshold=0, split_edges=0):
    q = gq()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), hub_threshold, split_edges)
    rp, co = g.rowptr.numpy(), g.col.numpy()
    H = synth.normal_matrix(g.n, d_in, seed=seed + 1)
    W = synth.glorot(d_in, d_out, seed=seed + 2)
    mask = synth.bernoulli_mask(g.n, mask_frac, seed=seed + 3)
    dY = synth.normal_matrix(g.n, d_out, seed=seed + 4, tag=synth.TAG_GRAD)
    sf, sb = synth.layer_seed(seed, 0, False), synth.layer_seed(seed, 0, True)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Hd, Wd, md, dYd = H.cuda(), W.cuda(), mask.cuda(), dY.cuda()
    A, Hout = q.gcn_layer_fwd(G, Hd, Wd, md, bits, sf, act, coef=coef, dev_err=err)
    dA = torch.empty(g.n, d_in, device="cuda")
    dW, dHin = q.gcn_layer_bwd(G, dYd, A, Hout, Wd, md, bits, sb, act, True, coef=coef, dA_save=dA, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    Hn, mn = H.numpy(), mask.numpy()
    pk = orc.quantize(Hn, mn, bits, sf) if bits < 32 else None
    A_ref = orc.spmm(rp, co, coef, orc.messages(Hn, pk, mn, d_in, bits))
    A_gpu = A.float().cpu().numpy()
    close(A_gpu, A_ref, rtol=5e-3, what="A (bf16)")
    Z = orc.gemm(A_gpu, W.numpy(), bf16=True)
    H_ref = np.maximum(Z, 0) if act else Z
    close(Hout.cpu().numpy(), H_ref, rtol=2e-2, what="H_out bar")
    close(Hout.cpu().numpy(), H_ref, rtol=1e-3, what="H_out")

    Hg = Hout.cpu().numpy()
    dZ = dY.numpy().astype(np.float64) * ((Hg > 0) if act else 1.0)
    dW_ref = orc.gemm(A_gpu.T, dZ, bf16=True)
    close(dW.cpu().numpy(), dW_ref, rtol=2e-2, what="dW bar")
    close(dW.cpu().numpy(), dW_ref, rtol=1e-3, what="dW")
    dA_ref = orc.gemm(dZ, W.numpy().T, bf16=True)
    dAg = dA.cpu().numpy()
    close(dAg, dA_ref, rtol=1e-3, what="dA")
    pkb = orc.quantize(dAg, mn, bits, sb) if bits < 32 else None
    dH_ref = orc.spmm(rp, co, coef, orc.messages(dAg, pkb, mn, d_in, bits), transpose=True)
    close(dHin.cpu().numpy(), dH_ref, rtol=1e-4, what="dH_in")


@pytest.mark.parametrize("bits", [2, 4, 8, 32])
@pytest.mark.parametrize("act", [0, 1])
def test_gcn_layer_tiny(orc, bits, act):
    # the tiny workload: uniform graph, 1,024 nodes, 64 -> 64, 30% marginal
    _case(orc, synth.uniform_graph(1024, 16384, seed=0), 64, 64, bits, act, coef=0)


@pytest.mark.parametrize("d_in,d_out", [(100, 256), (128, 256), (256, 256), (256, 47)])
@pytest.mark.parametrize("bits", [2, 8])
def test_gcn_layer_widths(orc, d_in, d_out, bits):
    _case(orc, rmat_small(), d_in, d_out, bits, act=1 if d_out != 47 else 0, coef=0, mask_frac=0.6)


@pytest.mark.parametrize("coef", [1, 2])
def test_gcn_layer_coefficients(orc, coef):
    _case(orc, rmat_small(), 64, 64, 4, 1, coef=coef, mask_frac=0.4)


def test_gcn_layer_hubs(orc):
    _case(orc, hub_graph(), 128, 128, 2, 1, coef=0, mask_frac=0.5, hub_threshold=40)
    _case(orc, hub_graph(), 128, 128, 2, 1, coef=0, mask_frac=0.5, hub_threshold=32, split_edges=256)


def test_gcn_layer_all_central_and_all_marginal(orc):
    _case(orc, rmat_small(), 64, 32, 8, 1, coef=0, mask_frac=0.0)
    _case(orc, rmat_small(), 64, 32, 8, 1, coef=0, mask_frac=1.0)


@pytest.mark.parametrize("bits", [2, 8, 32])
def test_gcn_layer_fused_dz_handoff(orc, bits):
    """The transposed aggregation writes the layer below's dZ = bf16(dH_in *
    [H_in > 0]) (the ReLU gate of the layer below, as the bits its forward
    wrote), and the layer below takes it as its dZ: dZ within the bf16 bar of
    the oracle's gated dH_in, and the layer below's dW from it at the GEMM
    bars."""
    q = gq()
    g = rmat_small()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda())
    rp, co = g.rowptr.numpy(), g.col.numpy()
    d0, d1, d2 = 100, 128, 64
    X = synth.normal_matrix(g.n, d0, seed=31)
    W0 = synth.glorot(d0, d1, seed=32)
    W1 = synth.glorot(d1, d2, seed=33)
    mask = synth.bernoulli_mask(g.n, 0.6, seed=34)
    dY = synth.normal_matrix(g.n, d2, seed=35, tag=synth.TAG_GRAD)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    md = mask.cuda()
    R0 = torch.empty(g.n, (d1 + 31) // 32, dtype=torch.int32, device="cuda")
    A0, H0 = q.gcn_layer_fwd(G, X.cuda(), W0.cuda(), md, bits, 1, q.ACT_RELU, dev_err=err, relu_bits=R0)
    A1, H1 = q.gcn_layer_fwd(G, H0, W1.cuda(), md, bits, 2, q.ACT_NONE, dev_err=err)
    dA1 = torch.empty(g.n, d1, device="cuda")
    dZ0 = torch.full((g.n, d1), float("nan"), dtype=torch.bfloat16, device="cuda")
    dW1, none = q.gcn_layer_bwd(G, dY.cuda(), A1, H1, W1.cuda(), md, bits, 3, q.ACT_NONE, True, dA_save=dA1,
                                dev_err=err, gate_in=R0, dZ_prev=dZ0)
    assert none is None
    dW0, _ = q.gcn_layer_bwd(G, None, A0, None, W0.cuda(), md, bits, 4, q.ACT_RELU, False, dev_err=err,
                             dZ_in=dZ0)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and int(G.status.cpu()[0]) == 0
    mn = mask.numpy()
    dAg = dA1.cpu().numpy()
    pkb = orc.quantize(dAg, mn, bits, 3) if bits < 32 else None
    dH = orc.spmm(rp, co, orc.COEF_GCN, orc.messages(dAg, pkb, mn, d1, bits), transpose=True)
    dZ_ref = dH * (H0.cpu().numpy() > 0)
    dZg = dZ0.float().cpu().numpy()
    close(dZg, dZ_ref, rtol=5e-3, what="fused dZ (bf16)")
    assert np.all(dZg[H0.cpu().numpy() <= 0] == 0.0)
    dW0_ref = orc.gemm(A0[:, :d0].float().cpu().numpy().T, dZg, bf16=True)
    close(dW0.cpu().numpy(), dW0_ref, rtol=2e-2, what="dW from the fused dZ bar")
    close(dW0.cpu().numpy(), dW0_ref, rtol=1e-3, what="dW from the fused dZ")


def _unpack_bits(words, d):
    """[n x d] bool from int32 words, bit c % 32 of word c // 32."""
    w = words.cpu().numpy().view(np.uint32)
    cols = np.arange(d)
    return ((w[:, cols // 32] >> (cols % 32).astype(np.uint32)) & 1).astype(bool)


@pytest.mark.parametrize("d_out", [16, 47, 100, 256])
@pytest.mark.parametrize("act", [0, 1])
def test_gcn_layer_relu_bits(d_out, act):
    """The forward's relu_bits are exactly [H_out > 0], bit c % 32 of word
    c // 32, with the bits past d_out clear."""
    q = gq()
    g = rmat_small()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda())
    d_in = 64
    X = synth.normal_matrix(g.n, d_in, seed=41).cuda()
    W = synth.glorot(d_in, d_out, seed=42).cuda()
    nw = (d_out + 31) // 32
    R = torch.full((g.n, nw + 1), -1, dtype=torch.int32, device="cuda")  # one word of padding per row
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, H = q.gcn_layer_fwd(G, X, W, None, 32, 1, act, dev_err=err, relu_bits=R)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = _unpack_bits(R[:, :nw], 32 * nw)
    np.testing.assert_array_equal(got[:, :d_out], H.cpu().numpy() > 0)
    assert not got[:, d_out:].any()
    assert bool((R[:, nw] == -1).all())  # words past ceil(d_out / 32) untouched
