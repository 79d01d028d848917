"""Pins of the oracle's message-level quantization metrics against facts
that do not come from the routines themselves:

  AdaQP Sec. 4.2 (Problem 11): the variance weight of a message row,
      beta_k = sum_{v in N_T(k)} a_{k,v}^2 * D * (max h_k - min h_k)^2 / 6,
  pinned by a hand-worked graph, by the aggregation of unit messages (the
  a_{k,v} are the entries the pinned SpMM applies) and by the variance the
  quantizer actually produces (beta_k / (2^b - 1)^2 is the variance of the
  aggregated quantization error of message k when its fractional parts are
  spread evenly);
  Tango Sec. 3.2 (Eq. 4): Error_X = (1/N) sum |X - Xq| / (|X| + |Xq| + eps),
  pinned by a hand-worked row, rows on the quantization grid, its range and
  its behaviour in the bit-width; and the bit-count rule built on it."""
import numpy as np
import pytest

import synth


def _tiny():
    # CSR by destination: 0 <- {0, 1}, 1 <- {1, 2}, 2 <- {2}
    return np.array([0, 2, 4, 5], np.int32), np.array([0, 1, 1, 2, 2], np.int32)


def test_beta_hand_example(orc):
    rp, co = _tiny()
    X = np.array([[0, 1], [0, 3], [1, 2]], np.float32)  # ranges 1, 3, 1; D = 2
    # deg_in = [2, 2, 1], deg_out = [1, 2, 2]; GCN a_{k,v} = 1/sqrt(deg_out(k) deg_in(v))
    #   node 0 -> 0: 1/2;  node 1 -> 0, 1: 1/4 + 1/4;  node 2 -> 1, 2: 1/4 + 1/2
    s2 = np.array([0.5, 0.5, 0.75])
    assert np.allclose(orc.beta(rp, co, orc.COEF_GCN, X), s2 * 2 * np.array([1, 9, 1]) / 6, rtol=1e-12)
    # GraphSAGE-mean a_{k,v} = 1/deg_in(v):  1/4;  1/4 + 1/4;  1/4 + 1
    s2 = np.array([0.25, 0.5, 1.25])
    assert np.allclose(orc.beta(rp, co, orc.COEF_SAGE, X), s2 * 2 * np.array([1, 9, 1]) / 6, rtol=1e-12)


@pytest.mark.parametrize("coef", [0, 1])
def test_beta_is_the_aggregation_of_unit_messages(orc, coef):
    g = synth.rmat_graph(scale=10, n=900, n_draws=900 * 8, seed=11)
    rp, co = g.rowptr.numpy(), g.col.numpy()
    X = synth.normal_matrix(g.n, 24, seed=5).numpy()
    beta = orc.beta(rp, co, coef, X)
    for k in (0, 1, 7, 300, 899):
        unit = np.zeros((g.n, 1))
        unit[k] = 1.0
        a = orc.spmm(rp, co, coef, unit)[:, 0]  # a[v] = a_{k,v}
        rng = float(X[k].max()) - float(X[k].min())
        assert beta[k] == pytest.approx((a ** 2).sum() * 24 * rng ** 2 / 6, rel=1e-12)


def test_beta_predicts_the_quantizers_variance(orc):
    # Message k = 0 with values j * 3/59 (j = 0..59): S = 1 at b = 2, and the
    # fractional parts run over the 59 multiples of 1/59 (59 is prime), so
    # the per-element variance p(1-p) S^2 averages to 1/6 up to 1/59^2.
    rp, co = _tiny()
    d, b = 60, 2
    x = (np.arange(d) * (3.0 / 59.0)).astype(np.float32)
    X = np.vstack([x, np.zeros(d, np.float32), np.zeros(d, np.float32)])
    beta = orc.beta(rp, co, orc.COEF_GCN, X)[0]
    T = 3000
    err2 = np.zeros(T)
    for s in range(T):
        deq = orc.dequant(orc.quantize(X[:1], None, b, 1000 + s), d, b)[0]
        err2[s] = ((deq.astype(np.float64) - x) ** 2).sum()
    # node 0 sends to node 0 only, with a^2 = 1/2
    measured = 0.5 * err2.mean()
    predicted = beta / (2 ** b - 1) ** 2
    assert measured == pytest.approx(predicted, rel=0.05)


def test_quant_error_hand_example(orc):
    # Row [0, 0.5, 1, 3] at b = 2: Z = 0, S = 1, so the codes of 0, 1 and 3
    # are exact and 0.5 becomes 0 or 1 by its stochastic-rounding uniform.
    X = np.array([[0.0, 0.5, 1.0, 3.0]], np.float32)
    for seed in (0, 1, 2, 3, 4, 5):
        pk = orc.quantize(X, None, 2, seed)
        q1 = 1 if 0.5 + orc.uniform(seed, 0, 1) >= 1.0 else 0
        assert list(orc.codes(pk, 4, 2)[0]) == [0, q1, 1, 3]
        eps = 5e-4
        expected = (0.5 / (0.5 + q1 + eps)) / 4
        assert orc.quant_error(X, pk, None, 2, eps) == pytest.approx(expected, rel=1e-12)


def test_quant_error_zero_on_the_grid(orc):
    # rows whose values are Z + q S exactly: no rounding error at all
    rng = np.random.default_rng(0)
    q = rng.integers(0, 16, size=(8, 32)).astype(np.float32)
    q[:, 0], q[:, 1] = 0, 15
    X = (q * 0.25 - 1.0).astype(np.float32)
    assert orc.quant_error(X, orc.quantize(X, None, 4, 3), None, 4) == 0.0


def test_quant_error_range_bits_and_mask(orc):
    X = synth.normal_matrix(200, 64, seed=2).numpy()
    errs = [orc.quant_error(X, orc.quantize(X, None, b, 9), None, b) for b in (2, 4, 8)]
    assert all(0.0 <= e <= 1.0 for e in errs)
    assert errs[0] > errs[1] > errs[2] > 0.0
    # rows left unquantized (mask 0) add zero terms but count in N
    mask = synth.bernoulli_mask(200, 0.5, seed=4).numpy()
    sel = mask.astype(bool)
    pk = orc.quantize(X, mask, 4, 9)
    e_mask = orc.quant_error(X, pk, mask, 4)
    e_sel = orc.quant_error(X[sel], pk[sel], None, 4)
    assert e_mask == pytest.approx(e_sel * sel.sum() / 200, rel=1e-12)


def test_bits_rule_picks_the_fewest_bits_under_threshold(orc):
    X = synth.normal_matrix(300, 64, seed=6).numpy()
    errs = {b: orc.quant_error(X, orc.quantize(X, None, b, 5), None, b) for b in (2, 4, 8)}
    for thr in (0.5, errs[2] + 1e-9, errs[2], errs[4], errs[8], 1e-9):
        b = orc.bits_for_error(X, None, 5, threshold=thr)
        ok = [c for c in (2, 4, 8) if errs[c] < thr]
        assert b == (ok[0] if ok else 8)


# --------------------------------------------------------------------------
# AdaQP Sec. 4.2, Problems 10-12 on one device: the per-row width choice
# --------------------------------------------------------------------------

def _objective(beta, bits, d, lam, gamma):
    L = (2.0 ** bits - 1.0)
    return lam * np.sum(beta / L ** 2) + (1 - lam) * gamma * np.sum(d * bits)


def test_assign_bits_extremes(orc):
    beta = np.array([0.0, 1e-6, 3.0, 5e4], np.float32)
    assert orc.assign_bits(beta, 64, 1.0, 1.0).tolist() == [2, 8, 8, 8]  # variance only; beta 0 ties to 2
    assert orc.assign_bits(beta, 64, 0.0, 1.0).tolist() == [2, 2, 2, 2]  # time only


def test_assign_bits_switch_points(orc):
    # the 2 -> 4 switch where lam beta (1/9 - 1/225) = (1 - lam) gamma d (4 - 2),
    # the 4 -> 8 switch where lam beta (1/225 - 1/65025) = (1 - lam) gamma d (8 - 4)
    d, lam, gamma = 32, 0.25, 0.5
    t24 = (1 - lam) * gamma * d * 2 / (lam * (1 / 9 - 1 / 225))
    t48 = (1 - lam) * gamma * d * 4 / (lam * (1 / 225 - 1 / 65025))
    beta = np.array([t24 * 0.99, t24 * 1.01, t48 * 0.99, t48 * 1.01], np.float32)
    assert orc.assign_bits(beta, d, lam, gamma).tolist() == [2, 4, 4, 8]


def test_assign_bits_minimizes_the_weighted_sum(orc):
    import itertools
    rng = np.random.default_rng(4)
    for trial in range(4):
        beta = (10.0 ** rng.uniform(0, 4, size=6)).astype(np.float32)
        d, lam, gamma = 16, float(rng.uniform(0.1, 0.9)), float(rng.uniform(0.1, 2.0))
        got = orc.assign_bits(beta, d, lam, gamma).astype(np.float64)
        best = min(_objective(beta.astype(np.float64), np.array(c, np.float64), d, lam, gamma)
                   for c in itertools.product((2, 4, 8), repeat=6))
        assert _objective(beta.astype(np.float64), got, d, lam, gamma) == pytest.approx(best, rel=1e-12)


def test_assign_bits_mask_and_the_mixed_pipeline(orc):
    # beta_k of a graph's messages -> widths -> the mixed-width quantizer
    g = synth.rmat_graph(scale=9, n=500, n_draws=500 * 8, seed=2)
    rp, co = g.rowptr.numpy(), g.col.numpy()
    X = synth.normal_matrix(g.n, 96, seed=7).numpy()
    beta = orc.beta(rp, co, orc.COEF_GCN, X).astype(np.float32)
    mask = synth.bernoulli_mask(g.n, 0.5, seed=1).numpy()
    rb = orc.assign_bits(beta, 96, 0.5, 1e-3, mask)
    assert set(np.unique(rb[mask == 0]).tolist()) == {0}
    assert set(np.unique(rb[mask == 1]).tolist()) <= {2, 4, 8}
    assert len(set(rb[mask == 1].tolist())) > 1  # this lam and gamma mix the widths
    pk, roff = orc.quantize_mixed(X, rb, 3)
    assert roff[-1] == sum(orc.pitch(96, int(b)) for b in rb if b in (2, 4, 8))
