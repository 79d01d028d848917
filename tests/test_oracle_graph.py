"""Pins of the oracle's aggregation and GCN layer against dense brute force
built from the pages' definitions (Sancus Sec. 2: A^ = D~^-1/2 (A+I) D~^-1/2;
AdaQP Sec. 2.1 weighted sum), closed forms and finite differences."""
import numpy as np
import pytest

import synth


def small_graph(n=40, m=160, seed=0, symmetric=False):
    g = synth.uniform_graph(n, m, seed=seed)
    rowptr, col = g.rowptr.numpy(), g.col.numpy()
    if symmetric:
        A = dense_adj(rowptr, col)
        A = np.maximum(A, A.T)
        rows, cols = np.nonzero(A)          # rows = destinations, sorted
        rowptr = np.zeros(n + 1, np.int32)
        np.add.at(rowptr, rows + 1, 1)
        rowptr = np.cumsum(rowptr).astype(np.int32)
        col = cols.astype(np.int32)
    return rowptr, col


def dense_adj(rowptr, col):
    """A_bar[v][u] = 1 for each CSR edge u -> v (self-loops are in the CSR)."""
    n = len(rowptr) - 1
    A = np.zeros((n, n))
    for v in range(n):
        A[v, col[rowptr[v]:rowptr[v + 1]]] = 1.0
    return A


def dense_gcn(rowptr, col):
    A = dense_adj(rowptr, col)
    din = A.sum(axis=1)          # row sums: in-degree incl. self-loop
    dout = A.sum(axis=0)         # column sums: out-degree incl. self-loop
    return np.diag(din ** -0.5) @ A @ np.diag(dout ** -0.5)


def test_graph_has_self_loops_and_sorted_rows():
    rowptr, col = small_graph()
    for v in range(len(rowptr) - 1):
        r = col[rowptr[v]:rowptr[v + 1]]
        assert v in r and np.all(np.diff(r) > 0)


def test_degree_norms_closed_form(orc):
    rowptr, col = small_graph(64, 400, seed=2)
    di, do, ii = orc.degree_norms(rowptr, col)
    A = dense_adj(rowptr, col)
    din, dout = A.sum(1), A.sum(0)
    assert np.all(np.abs(di.astype(np.float64) ** 2 * din - 1) < 2 ** -21)
    assert np.all(np.abs(do.astype(np.float64) ** 2 * dout - 1) < 2 ** -21)
    assert np.all(np.abs(ii.astype(np.float64) * din - 1) < 2 ** -23)
    # perfect squares are exact
    for deg, want in ((1, 1.0), (4, 0.5), (16, 0.25), (64, 0.125)):
        sel = din == deg
        assert np.all(di[sel] == np.float32(want))


@pytest.mark.parametrize("symmetric", [False, True])
def test_spmm_gcn_dense_bruteforce(orc, symmetric):
    rowptr, col = small_graph(48, 300, seed=5, symmetric=symmetric)
    n = len(rowptr) - 1
    M = np.random.default_rng(0).standard_normal((n, 7))
    Ahat = dense_gcn(rowptr, col)
    np.testing.assert_allclose(orc.spmm(rowptr, col, orc.COEF_GCN, M), Ahat @ M, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(orc.spmm(rowptr, col, orc.COEF_GCN, M, transpose=True), Ahat.T @ M,
                               rtol=1e-12, atol=1e-12)
    if symmetric:
        # textbook: A^ D~^{1/2} 1 = D~^{1/2} 1 for the symmetric normalization
        s = np.sqrt(dense_adj(rowptr, col).sum(1))[:, None]
        np.testing.assert_allclose(orc.spmm(rowptr, col, orc.COEF_GCN, s), s, rtol=1e-12)
        w = np.linalg.eigvalsh(Ahat)
        assert w.max() < 1 + 1e-9 and w.min() > -1 - 1e-9


def test_spmm_sage_mean(orc):
    rowptr, col = small_graph(48, 300, seed=6)
    n = len(rowptr) - 1
    ones = np.ones((n, 3))
    np.testing.assert_allclose(orc.spmm(rowptr, col, orc.COEF_SAGE, ones), ones, rtol=1e-14)
    M = np.random.default_rng(1).standard_normal((n, 5))
    A = dense_adj(rowptr, col)
    mean = (A / A.sum(1, keepdims=True)) @ M
    np.testing.assert_allclose(orc.spmm(rowptr, col, orc.COEF_SAGE, M), mean, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(orc.spmm(rowptr, col, orc.COEF_ONE, M), A @ M, rtol=1e-12, atol=1e-12)


def test_spmm_adjoint(orc):
    rowptr, col = small_graph(60, 500, seed=7)
    n = len(rowptr) - 1
    rng = np.random.default_rng(2)
    X, G = rng.standard_normal((n, 4)), rng.standard_normal((n, 4))
    for coef in (orc.COEF_GCN, orc.COEF_SAGE):
        lhs = np.sum(orc.spmm(rowptr, col, coef, X) * G)
        rhs = np.sum(X * orc.spmm(rowptr, col, coef, G, transpose=True))
        assert abs(lhs - rhs) < 1e-10 * (1 + abs(lhs))


def test_messages_mix_mask(orc):
    X = synth.normal_matrix(30, 16, seed=1).numpy()
    mask = synth.bernoulli_mask(30, 0.5, seed=4).numpy()
    pk = orc.quantize(X, mask, 4, 3)
    M = orc.messages(X, pk, mask, 16, 4)
    np.testing.assert_array_equal(M[mask == 0], X[mask == 0])
    deq = orc.dequant(orc.quantize(X, None, 4, 3), 16, 4)
    np.testing.assert_array_equal(M[mask == 1], deq[mask == 1])


def test_bf16_round_closed_form(orc):
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 2 ** -7, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38], np.float32)
    want = np.array([1.0, 1.0, 1.0 + 2 ** -7, 1.0 + 2 ** -6, -2.5, 2.9967e38], np.float32)
    got = orc.bf16_round(x)
    np.testing.assert_array_equal(got[:5], want[:5])       # ties to even at 1+2^-8, 1+3*2^-8
    assert abs(got[5] / want[5] - 1) < 2 ** -8


def _loss_fwd(orc, rowptr, col, coef, H, W, relu, G):
    o = orc.gcn_layer_fwd(rowptr, col, coef, H, W, None, 32, 0, relu, bf16=False)
    return np.sum(o["H_out"] * G), o


@pytest.mark.parametrize("coef,relu", [(0, True), (1, False)])
def test_gcn_layer_finite_differences(orc, coef, relu):
    rowptr, col = small_graph(30, 150, seed=8)
    n = len(rowptr) - 1
    rng = np.random.default_rng(3)
    H = rng.standard_normal((n, 6)).astype(np.float32)
    W = rng.standard_normal((6, 5))
    G = rng.standard_normal((n, 5))
    L0, o = _loss_fwd(orc, rowptr, col, coef, H, W, relu, G)
    b = orc.gcn_layer_bwd(rowptr, col, coef, G, o["A"], o["Z"], W, None, 32, 0, relu, bf16=False)
    h = 1e-3
    for (i, j) in [(0, 0), (3, 4), (5, 2)]:
        Wp, Wm = W.copy(), W.copy()
        Wp[i, j] += h
        Wm[i, j] -= h
        fd = (_loss_fwd(orc, rowptr, col, coef, H, Wp, relu, G)[0]
              - _loss_fwd(orc, rowptr, col, coef, H, Wm, relu, G)[0]) / (2 * h)
        assert abs(fd - b["dW"][i, j]) < 1e-6 * (1 + abs(fd))
    # H is fp32 in the layer interface: use a step that is exact in fp32
    hh = 2.0 ** -6
    for (i, j) in [(0, 1), (7, 3), (20, 5)]:
        Hp, Hm = H.copy(), H.copy()
        Hp[i, j] += hh
        Hm[i, j] -= hh
        fd = (_loss_fwd(orc, rowptr, col, coef, Hp, W, relu, G)[0]
              - _loss_fwd(orc, rowptr, col, coef, Hm, W, relu, G)[0]) / (2 * hh)
        assert abs(fd - b["dH_in"][i, j]) < 1e-3 * (1 + abs(fd))


def test_gcn_quantized_forward_unbiased(orc):
    # linearity + Eqn 6: the expectation over seeds of the quantized
    # aggregation equals the unquantized aggregation.
    rowptr, col = small_graph(24, 100, seed=9)
    n = len(rowptr) - 1
    X = synth.normal_matrix(n, 8, seed=2).numpy()
    mask = synth.bernoulli_mask(n, 0.5, seed=3).numpy()
    ref = orc.spmm(rowptr, col, 0, X.astype(np.float64))
    T = 2048
    acc = np.zeros_like(ref)
    for s in range(T):
        pk = orc.quantize(X, mask, 2, s)
        acc += orc.spmm(rowptr, col, 0, orc.messages(X, pk, mask, 8, 2))
    S, _ = orc.header(orc.quantize(X, None, 2, 0), 8, 2)
    assert np.max(np.abs(acc / T - ref)) < 5 * S.max() / (2 * np.sqrt(T))
