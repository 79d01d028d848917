"""Message-level quantization metrics on the GPU vs the oracle:
AdaQP Sec. 4.2 beta_k (gq_message_variance_weights) and Tango Sec. 3.2
Eq. 4 Error_X (gq_quant_error) with its bit-count rule.  beta within
1e-4 (1 + |ref|) relative to the oracle's float64 value; Error_X on the
GPU's own packed bytes within 1e-5 relative."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import gq, hub_graph, rmat_small, sparse_rows_graph

pytestmark = pytest.mark.gpu


def _rel_close(gpu, ref, rtol):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref) - rtol * np.maximum(np.abs(ref), 1e-30)
    assert err.max() <= 0, (float(np.abs(gpu - ref).max()), int((err > 0).sum()))


@pytest.mark.parametrize("graph", ["uniform", "rmat", "hubs", "hubs_split", "sparse_rows"])
@pytest.mark.parametrize("coef", [0, 1, 2])
@pytest.mark.parametrize("d", [7, 64, 256])
def test_beta(orc, graph, coef, d):
    q = gq()
    g = {"uniform": lambda: synth.uniform_graph(1024, 16384, seed=0), "rmat": rmat_small,
         "hubs": hub_graph, "hubs_split": hub_graph, "sparse_rows": sparse_rows_graph}[graph]()
    kw = dict(hub_threshold=32, split_edges=256) if graph == "hubs_split" else {}
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), **kw)
    if graph == "hubs_split":
        assert G.c.tr_sched.n_groups > 0  # nodes whose out-edges are cut into several tasks
    X = synth.normal_matrix(g.n, d, seed=d + coef).numpy()
    beta = q.message_variance_weights(G, torch.from_numpy(X).cuda(), coef).cpu().numpy()
    _rel_close(beta, orc.beta(g.rowptr.numpy(), g.col.numpy(), coef, X), 1e-4)


def test_beta_padded_rows(orc):
    q = gq()
    g = rmat_small()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda())
    Xfull = synth.normal_matrix(g.n, 40, seed=3)
    X = Xfull[:, :33]  # ldx = 40 > d = 33
    beta = q.message_variance_weights(G, Xfull.cuda()[:, :33], 0).cpu().numpy()
    _rel_close(beta, orc.beta(g.rowptr.numpy(), g.col.numpy(), 0, X.contiguous().numpy()), 1e-4)


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("d", [5, 64, 100, 256])
@pytest.mark.parametrize("mask_frac", [None, 0.4])
def test_quant_error(orc, bits, d, mask_frac):
    q = gq()
    n = 3000
    X = synth.normal_matrix(n, d, seed=bits * 7 + d).numpy()
    mask = None if mask_frac is None else synth.bernoulli_mask(n, mask_frac, seed=2).numpy()
    Xd = torch.from_numpy(X).cuda()
    md = None if mask is None else torch.from_numpy(mask).cuda()
    pk = q.quantize_pack(Xd, md, bits, 17)
    err = float(q.quant_error(Xd, pk, md, bits).item())
    ref = orc.quant_error(X, pk.cpu().numpy(), mask, bits)
    assert err == pytest.approx(ref, rel=1e-5)
    assert 0.0 <= err <= 1.0


def test_quant_error_empty_and_constant_rows(orc):
    q = gq()
    X0 = torch.zeros(0, 16, device="cuda")
    pk = q.quantize_pack(X0, None, 4, 1)
    assert float(q.quant_error(X0, pk, None, 4).item()) == 0.0
    X = np.full((10, 16), 2.5, np.float32)  # constant rows de-quantize exactly
    Xd = torch.from_numpy(X).cuda()
    assert float(q.quant_error(Xd, q.quantize_pack(Xd, None, 2, 1), None, 2).item()) == 0.0


@pytest.mark.parametrize("n,d,mask_frac", [(2000, 64, None), (777, 100, 0.5), (300, 1000, 0.8), (64, 3, None)])
def test_bits_rule_matches_oracle(orc, n, d, mask_frac):
    """Tango Sec. 3.2: the one-pass rule (gq_bits_for_error) gives the
    oracle's Error_X at 2, 4 and 8 bits (1e-5 relative) and, wherever the
    threshold is not within 1e-4 of an error, the oracle's choice of bits."""
    q = gq()
    X = synth.normal_matrix(n, d, seed=8 + d).numpy()
    mask = None if mask_frac is None else synth.bernoulli_mask(n, mask_frac, seed=3).numpy()
    Xd = torch.from_numpy(X).cuda()
    md = None if mask is None else torch.from_numpy(mask).cuda()
    errs = {b: orc.quant_error(X, orc.quantize(X, mask, b, 5), mask, b) for b in (2, 4, 8)}
    e3 = torch.empty(3, dtype=torch.float64, device="cuda")
    thrs = (0.5, errs[2] * 0.999, errs[2] * 1.001, errs[4] * 1.001, errs[4] * 0.999, errs[8] * 1.001, 1e-6)
    for thr in thrs:
        b = int(q.bits_for_error(Xd, md, 5, threshold=thr, err3=e3).item())
        assert e3.cpu().numpy() == pytest.approx([errs[2], errs[4], errs[8]], rel=1e-5)
        if all(abs(errs[k] - thr) > 1e-4 * thr for k in (2, 4, 8)):
            assert b == orc.bits_for_error(X, mask, 5, threshold=thr), thr
    # the same errors as gq_quant_error on the quantizer's own packed rows
    for i, bb in enumerate((2, 4, 8)):
        pk = q.quantize_pack(Xd, md, bb, 5)
        assert float(q.quant_error(Xd, pk, md, bb).item()) == pytest.approx(float(e3[i].item()), rel=1e-6)


def test_bits_rule_empty_and_constant(orc):
    q = gq()
    X0 = torch.zeros(0, 16, device="cuda")
    e3 = torch.empty(3, dtype=torch.float64, device="cuda")
    assert int(q.bits_for_error(X0, None, 1, err3=e3).item()) == 2 and float(e3.abs().max()) == 0.0
    Xc = torch.full((10, 16), 2.5, device="cuda")  # constant rows: no error at any width
    assert int(q.bits_for_error(Xc, None, 1, err3=e3).item()) == 2 and float(e3.abs().max()) == 0.0
    with pytest.raises(q.GQError):
        q.bits_for_error(Xc, None, 1, threshold=0.0)
    with pytest.raises(q.GQError):
        q.bits_for_error(Xc, None, 1, eps=0.0)


def test_quant_error_rejects_bad_arguments():
    q = gq()
    X = torch.zeros(4, 8, device="cuda")
    pk = q.quantize_pack(X, None, 4, 0)
    with pytest.raises(q.GQError):
        q.quant_error(X, pk, None, 3)
    with pytest.raises(q.GQError):
        q.quant_error(X, pk, None, 4, eps=0.0)


# AdaQP Sec. 4.2 Problems 10-12 on one device: per-row widths, bit-exact
@pytest.mark.parametrize("lam,gamma", [(0.5, 1e-3), (0.25, 0.5), (1.0, 1.0), (0.0, 1.0), (0.9, 1e-6)])
def test_assign_bits(orc, lam, gamma):
    q = gq()
    rng = np.random.default_rng(11)
    d = 64
    beta = (10.0 ** rng.uniform(-3, 7, size=20000)).astype(np.float32)
    if 0 < lam < 1:  # values just either side of the 2/4 and 4/8 switch points
        t24 = (1 - lam) * gamma * d * 2 / (lam * (1 / 9 - 1 / 225))
        t48 = (1 - lam) * gamma * d * 4 / (lam * (1 / 225 - 1 / 65025))
        beta[:6] = np.array([t24 * (1 - 1e-6), t24, t24 * (1 + 1e-6), t48 * (1 - 1e-6), t48, t48 * (1 + 1e-6)])
    beta[6] = 0.0
    mask = synth.bernoulli_mask(beta.size, 0.7, seed=3).numpy()
    for m in (None, mask):
        got = q.assign_bits(torch.from_numpy(beta).cuda(), d, lam, gamma,
                            None if m is None else torch.from_numpy(m).cuda()).cpu().numpy()
        np.testing.assert_array_equal(got, orc.assign_bits(beta, d, lam, gamma, m))


def test_assign_bits_empty_and_arguments():
    q = gq()
    assert q.assign_bits(torch.zeros(0, device="cuda"), 8, 0.5, 1.0).numel() == 0
    b = torch.ones(4, device="cuda")
    for lam, gamma in ((1.5, 1.0), (-0.1, 1.0), (0.5, -1.0), (0.5, float("nan"))):
        with pytest.raises(q.GQError):
            q.assign_bits(b, 8, lam, gamma)


def test_beta_to_widths_to_mixed_aggregation(orc):
    # the whole adaptive path on the GPU: beta -> widths -> mixed quantization
    # -> mixed aggregation, checked against the oracle on the GPU's widths
    q = gq()
    g = rmat_small()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda())
    d = 128
    X = synth.normal_matrix(g.n, d, seed=21).numpy()
    Xd = torch.from_numpy(X).cuda()
    mask = synth.bernoulli_mask(g.n, 0.6, seed=4).cuda()
    beta = q.message_variance_weights(G, Xd, 0)
    rb = q.assign_bits(beta, d, 0.5, 2e-3, mask)
    rbh = rb.cpu().numpy()
    np.testing.assert_array_equal(rbh, orc.assign_bits(beta.cpu().numpy(), d, 0.5, 2e-3, mask.cpu().numpy()))
    assert len(set(rbh.tolist())) >= 3  # full-precision rows and at least two widths
    pk, roff = q.quantize_pack_mixed(Xd, rb, 8)
    Y = q.dequant_spmm_mixed(G, Xd, pk, roff, rb, coef=0).cpu().numpy()
    M = orc.messages_mixed(X, pk.cpu().numpy(), roff.cpu().numpy(), rbh, d)
    from gpu_helpers import close
    close(Y, orc.spmm(g.rowptr.numpy(), g.col.numpy(), 0, M), what="beta -> widths -> aggregation")
