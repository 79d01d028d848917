"""Pins of the oracle's row-list forms, which the parity tests at the
largest sizes use: the quantizer on a list of rows (AdaQP Sec. 2.3, Eqn 4,
the noise keyed by each row's node id) and the aggregation evaluated at a
list of output rows (AdaQP Sec. 2.1 weighted sum with Sancus Sec. 2's
normalized adjacency).  Each is held against dense brute force of the
definition on a small graph, and against the whole-matrix routines."""
import numpy as np
import pytest

import synth
from test_oracle_graph import dense_adj, dense_gcn


def _graph(seed=4):
    g = synth.rmat_graph(scale=8, n=200, n_draws=200 * 10, seed=seed)
    return g.rowptr.numpy(), g.col.numpy()


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_quantize_rows_match_whole_matrix(orc, bits):
    X = synth.normal_matrix(300, 37 * 4, seed=9).numpy()
    ids = np.array([0, 1, 5, 77, 150, 299], np.int64)
    whole = orc.quantize(X, None, bits, 1234)
    np.testing.assert_array_equal(orc.quantize_rows(X[ids], ids, bits, 1234), whole[ids])
    # the node id keys the noise: the same values under other ids code differently
    other = orc.quantize_rows(X[ids], ids + 1, bits, 1234)
    assert not np.array_equal(other, whole[ids])


@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("coef", [0, 1, 2])
def test_spmm_rows_dense_brute_force(orc, coef, transpose):
    rowptr, col = _graph()
    n = len(rowptr) - 1
    d = 6
    M = np.random.default_rng(1).standard_normal((n, d))
    A = dense_adj(rowptr, col)
    if coef == 0:
        Ahat = dense_gcn(rowptr, col)
    elif coef == 1:
        Ahat = A / A.sum(axis=1, keepdims=True)
    else:
        Ahat = A
    full = (Ahat.T if transpose else Ahat) @ M
    rows = np.array([0, 3, 17, 64, 150, n - 1], np.int64)
    ids = np.arange(n, dtype=np.int64)
    Y = orc.spmm_rows(rowptr, col, coef, rows, ids, M, transpose=transpose)
    np.testing.assert_allclose(Y, full[rows], rtol=1e-12, atol=1e-12)
    # the whole-matrix routine agrees at the same rows
    np.testing.assert_allclose(Y, orc.spmm(rowptr, col, coef, M, transpose=transpose)[rows], rtol=1e-12,
                               atol=1e-12)


@pytest.mark.parametrize("transpose", [False, True])
def test_spmm_rows_with_only_the_needed_messages(orc, transpose):
    rowptr, col = _graph(seed=6)
    n = len(rowptr) - 1
    M = np.random.default_rng(2).standard_normal((n, 5))
    rows = np.array([2, 40, 41, 199], np.int64)
    A = dense_adj(rowptr, col)
    need = np.nonzero((A[:, rows] if transpose else A[rows, :]).sum(axis=1 if transpose else 0))[0]
    Y = orc.spmm_rows(rowptr, col, 0, rows, need, M[need], transpose=transpose)
    ref = (dense_gcn(rowptr, col).T if transpose else dense_gcn(rowptr, col)) @ M
    np.testing.assert_allclose(Y, ref[rows], rtol=1e-12, atol=1e-12)
    # a missing message row is an error, not a silent zero
    with pytest.raises(ValueError):
        orc.spmm_rows(rowptr, col, 0, rows, need[1:], M[need[1:]], transpose=transpose)
