"""Parity at the largest sizes, in the launch configurations `bench.py`
times, on sampled rows (each output row depends only on its own edges, so
the oracle computes it alone, with coefficients from the whole graph's
degrees):
  - the large power-law GCN workload (2,449,029 nodes, 64.3M edges with
    self-loops, 100 -> 256 -> 256 -> 47, 60% marginal, b = 2) through the
    3-layer stack the benchmark times (model.GCNStack), every layer forward
    and backward, teacher-forced on the GPU's own stage inputs: A (bf16
    store, 5e-3), H_out (bf16 GEMM inputs: 2e-2 bar, 1e-3 checked), dW over
    all rows, dA, and the layer below's dZ that the transposed aggregation
    writes (its dH_in with the ReLU gate, bf16 store: 5e-3), on sampled rows
    including the heaviest;
  - the aggregation on the largest graph (16,777,216 nodes, ~537M edges,
    d = 256, b = 8, every row packed: 4.6 GB of packed rows, above 4 GiB),
    forward and transposed, with the quantized bytes of every row read
    bit-exact and the outputs within 1e-4 (1 + |ref|), on sampled rows
    including the heaviest and the last ids.
AdaQP Sec. 2.1 / 2.3 (Eqn 4-5) / 3.1; Sancus Sec. 2."""
import numpy as np
import pytest
import torch

import synth
from synth.configs import AGG_SWEEP, GCN3_LARGE
from gpu_helpers import close, gq, sample_rows

pytestmark = pytest.mark.gpu


def _in_sources(rp, co, rows):
    """Distinct sources of the in-edges of `rows` (ascending)."""
    return np.unique(np.concatenate([co[rp[v]:rp[v + 1]] for v in rows]))


def _out_targets(rp, co, rows, n):
    """Distinct destinations of the out-edges of `rows` (ascending)."""
    flag = np.zeros(n, bool)
    flag[rows] = True
    deg = np.diff(rp)
    dst = np.repeat(np.arange(n, dtype=np.int64), deg)
    return np.unique(dst[flag[co]])


def _messages(orc, Xd, ids, mask, d, bits, seed):
    """Message rows of nodes `ids` from the GPU matrix Xd: quantized by the
    oracle at their node ids where marginal (bits < 32), else the fp32 row."""
    Xr = Xd[torch.from_numpy(ids).to(Xd.device)].cpu().numpy()
    mk = np.ones(ids.size, np.uint8) if mask is None else mask[ids]
    pk = np.zeros((ids.size, orc.pitch(d, bits)), np.uint8) if bits < 32 else None
    if bits < 32 and mk.any():
        sel = np.nonzero(mk)[0]
        pk[sel] = orc.quantize_rows(Xr[sel], ids[sel], bits, seed)
    return orc.messages(Xr, pk, mk, d, bits), pk, mk


def test_large_gcn_stack_sampled(orc):
    q = gq()
    from quantized_gnn_message_gb300.model import GCNStack
    w = GCN3_LARGE
    g = w.make_graph(device="cuda")
    G = q.graph_prepare(g.rowptr, g.col)
    widths = w.widths
    L = len(widths) - 1
    X = synth.normal_matrix(g.n, widths[0], seed=w.seed, device="cuda")
    Ws = [synth.glorot(widths[l], widths[l + 1], seed=w.seed + 1 + l, device="cuda") for l in range(L)]
    maskd = synth.bernoulli_mask(g.n, w.mask_frac, seed=w.seed, device="cuda")
    dY = synth.normal_matrix(g.n, widths[-1], seed=w.seed, tag=synth.TAG_GRAD, device="cuda")
    bits = w.bits[0]
    sf = [synth.layer_seed(w.seed ^ (bits << 56), l, False) for l in range(L)]
    sb = [synth.layer_seed(w.seed ^ (bits << 56), l, True) for l in range(L)]
    model = GCNStack(G, widths, maskd, keep_dA=True)
    model.forward(X, Ws, bits, sf)
    model.backward(dY, Ws, bits, sb)
    torch.cuda.synchronize()
    assert int(model.err.item()) == 0 and int(G.status.cpu()[0]) == 0

    rp, co = g.rowptr.cpu().numpy(), g.col.cpu().numpy()
    n = g.n
    mask = maskd.cpu().numpy()
    rows = sample_rows(rp, 48, seed=11, n_heavy=6)
    rows_out = sample_rows(np.concatenate([[0], np.cumsum(np.bincount(co, minlength=n))]), 48, seed=12, n_heavy=6)
    ridx = torch.from_numpy(rows).cuda()
    oidx = torch.from_numpy(rows_out).cuda()
    H_in = X
    for l in range(L):
        d_in = widths[l]
        src = _in_sources(rp, co, rows)
        M, _, _ = _messages(orc, H_in, src, mask, d_in, bits, sf[l])
        A_ref = orc.spmm_rows(rp, co, orc.COEF_GCN, rows, src, M)
        A_gpu = model.A[l][:, :d_in][ridx].float().cpu().numpy()
        close(A_gpu, A_ref, rtol=5e-3, what=f"layer {l} A (bf16)")
        Z = orc.gemm(A_gpu, Ws[l].cpu().numpy(), bf16=True)
        H_ref = np.maximum(Z, 0) if l < L - 1 else Z
        Hg = model.H[l][ridx].cpu().numpy()
        close(Hg, H_ref, rtol=2e-2, what=f"layer {l} H_out bar")
        close(Hg, H_ref, rtol=1e-3, what=f"layer {l} H_out")
        H_in = model.H[l]

    # the stack's backward is fused: the transposed aggregation of layer l
    # writes layer l-1's dZ (bf16, ReLU gate applied), which layer l-1 takes
    assert model.fuse_dz
    for l in reversed(range(L)):
        d_in = widths[l]
        Wn = Ws[l].cpu().numpy()
        # dW over every row (a reduction over the whole graph)
        A_all = model.A[l][:, :d_in].float().cpu().numpy()
        dZ_all = (dY if l == L - 1 else model.dZ[l]).float().cpu().numpy().astype(np.float64)[:, :widths[l + 1]]
        dW_ref = orc.gemm(A_all.T, dZ_all, bf16=True)
        close(model.dW[l].cpu().numpy(), dW_ref, rtol=2e-2, what=f"layer {l} dW bar")
        # a sum over 2.45M rows whose terms largely cancel: fp32 accumulation
        # is held to 2^-20 of the sum of the terms' magnitudes
        mag = orc.gemm(np.abs(A_all).T, np.abs(dZ_all), bf16=True)
        del A_all
        err = np.abs(model.dW[l].cpu().numpy() - dW_ref) - (1e-3 * (1 + np.abs(dW_ref)) + 2.0 ** -20 * mag)
        assert err.max() <= 0, f"layer {l} dW: {int((err > 0).sum())} entries beyond the fp32 accumulation bound"
        if l == 0:
            break
        dA_ref = orc.gemm(dZ_all[rows], Wn.T, bf16=True)
        del dZ_all
        close(model.dA[l][ridx].cpu().numpy(), dA_ref, rtol=1e-3, what=f"layer {l} dA")
        # transposed aggregation of dA's messages (marginal rows quantized with the backward seed)
        dst = _out_targets(rp, co, rows_out, n)
        M, _, _ = _messages(orc, model.dA[l], dst, mask, d_in, bits, sb[l])
        dH_ref = orc.spmm_rows(rp, co, orc.COEF_GCN, rows_out, dst, M, transpose=True)
        gate = model.H[l - 1][oidx].cpu().numpy() > 0
        dZg = model.dZ[l - 1][oidx].float().cpu().numpy()[:, :d_in]
        close(dZg, dH_ref * gate, rtol=5e-3, what=f"layer {l - 1} dZ (bf16, from layer {l}'s dH_in)")
        assert np.all(dZg[~gate] == 0.0)


def test_largest_aggregation_sampled(orc):
    q = gq()
    w = AGG_SWEEP
    d, bits, seed = 256, 8, 7
    g = w.make_graph(device="cuda")
    G = q.graph_prepare(g.rowptr, g.col)
    n = g.n
    X = synth.normal_matrix(n, d, seed=w.seed, device="cuda")
    pk = q.quantize_pack(X, None, bits, seed)
    assert pk.numel() > (4 << 30)
    rp, co = g.rowptr.cpu().numpy(), g.col.cpu().numpy()
    rows = np.unique(np.concatenate([sample_rows(rp, 40, seed=21, n_heavy=6), [n - 2, n - 1]]))
    outdeg = np.bincount(co, minlength=n)
    rows_t = np.unique(np.concatenate([sample_rows(np.concatenate([[0], np.cumsum(outdeg)]), 40, seed=22,
                                                   n_heavy=6), [n - 1]]))
    pk_rows = lambda ids: pk[torch.from_numpy(ids).cuda()].cpu().numpy()
    for transpose, out_rows in ((False, rows), (True, rows_t)):
        Y = q.dequant_spmm(G, None, pk, None, d, bits, coef=q.COEF_GCN, transpose=transpose)
        torch.cuda.synchronize()
        assert int(G.status.cpu()[0]) == 0
        ids = _out_targets(rp, co, out_rows, n) if transpose else _in_sources(rp, co, out_rows)
        M, pk_ref, _ = _messages(orc, X, ids, None, d, bits, seed)
        np.testing.assert_array_equal(pk_rows(ids), pk_ref)      # every row read, bit for bit
        M_gpu = orc.messages(np.zeros((ids.size, d), np.float32), pk_rows(ids), None, d, bits)
        Y_ref = orc.spmm_rows(rp, co, orc.COEF_GCN, out_rows, ids, M_gpu, transpose=transpose)
        close(Y[torch.from_numpy(out_rows).cuda()].cpu().numpy(), Y_ref, what=f"transpose={transpose}")
        del Y
        torch.cuda.empty_cache()
