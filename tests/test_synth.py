"""The seeded input generators both sides draw their inputs from: their
counter hash equals the oracle's (each written independently from the
published MurmurHash3 finalizer), they are deterministic per seed, their
graphs are valid CSR by destination with one self-loop per node, and their
dense draws have the stated distributions."""
import math

import numpy as np
import torch

import synth


def test_hash_matches_the_oracle(orc):
    rng = np.random.default_rng(0)
    for seed in (0, 1, 0xDEADBEEFCAFE, 2 ** 63 + 5):
        rows = rng.integers(0, 2 ** 31, size=300)
        cols = rng.integers(0, 2 ** 20, size=300)
        got = synth.hash_u32(seed, torch.from_numpy(rows), torch.from_numpy(cols)).numpy()
        assert got.tolist() == [orc.hash32(seed, int(r), int(c)) for r, c in zip(rows, cols)]


def _check_csr(g):
    rp, col = g.rowptr.numpy().astype(np.int64), g.col.numpy()
    assert rp[0] == 0 and rp[-1] == col.size == g.nnz and np.all(np.diff(rp) >= 0)
    assert col.min() >= 0 and col.max() < g.n
    for v in range(g.n):
        r = col[rp[v]:rp[v + 1]]
        assert np.all(np.diff(r) > 0) and v in r  # ascending, distinct, with the self-loop


def test_rmat_deterministic_valid_and_heavy_tailed():
    a = synth.rmat_graph(scale=12, n=3000, n_draws=36000, seed=4)
    b = synth.rmat_graph(scale=12, n=3000, n_draws=36000, seed=4)
    c = synth.rmat_graph(scale=12, n=3000, n_draws=36000, seed=5)
    assert torch.equal(a.rowptr, b.rowptr) and torch.equal(a.col, b.col)
    assert a.col.numel() != c.col.numel() or not torch.equal(a.col, c.col)
    _check_csr(a)
    deg = np.diff(a.rowptr.numpy())
    assert deg.max() > 10 * deg.mean()


def test_rmat_exact_edge_count():
    g = synth.rmat_graph(scale=11, n=2000, n_draws=2000 * 4, seed=1, exact_edges=2000 * 6)
    assert g.nnz == 2000 * 6 + 2000  # the distinct pairs kept, plus one self-loop per node
    _check_csr(g)


def test_uniform_graph_valid():
    _check_csr(synth.uniform_graph(1024, 16384, seed=0))


def test_normal_matrix_moments_and_stream_rows():
    X = synth.normal_matrix(4096, 256, seed=3).numpy().astype(np.float64)
    assert abs(X.mean()) < 4 / math.sqrt(X.size) and abs(X.std() - 1) < 0.01
    assert np.array_equal(synth.normal_matrix(10, 256, seed=3, row0=100).numpy(), X[100:110].astype(np.float32))
    assert not np.array_equal(synth.normal_matrix(10, 256, seed=3, tag=synth.TAG_GRAD).numpy(),
                              X[:10].astype(np.float32))


def test_glorot_range_and_variance():
    W = synth.glorot(256, 128, seed=2).numpy().astype(np.float64)
    r = math.sqrt(6 / 384)
    assert np.all(np.abs(W) <= r) and abs(W.var() - r * r / 3) < 0.05 * r * r / 3


def test_bernoulli_mask_fraction():
    for f in (0.0, 0.3, 0.6, 1.0):
        m = synth.bernoulli_mask(200000, f, seed=9).numpy()
        assert set(np.unique(m).tolist()) <= {0, 1}
        assert abs(m.mean() - f) <= 4 * math.sqrt(f * (1 - f) / m.size) + 1e-12


def test_quantization_site_seeds_are_distinct():
    seeds = {synth.layer_seed(7, l, bw, w) for l in range(4) for bw in (False, True) for w in range(3)}
    assert len(seeds) == 24
