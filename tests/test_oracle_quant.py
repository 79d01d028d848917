"""Pins of the oracle's quantizer (AdaQP Sec. 2.3, Eqn 4-6) against facts
that do not come from the oracle itself: hand-worked packed bytes, the
published MurmurHash3 test vectors, the exact error bound, the rounding
probability, unbiasedness and the variance bound."""
import json
import math
import os

import numpy as np
import pytest

import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_fmix32_published_vectors(orc):
    # MurmurHash3_x86_32 of the empty input with seed s is fmix32(s); its
    # published test vectors are 0 -> 0, 1 -> 0x514E28B7, 0xFFFFFFFF -> 0x81F16F39.
    assert orc.fmix32(0) == 0
    assert orc.fmix32(1) == 0x514E28B7
    assert orc.fmix32(0xFFFFFFFF) == 0x81F16F39


def test_uniform_range_and_grid(orc):
    us = np.array([orc.uniform(12345, r, c) for r in range(64) for c in range(64)])
    assert us.min() >= 0.0 and us.max() <= 1.0 - 2.0 ** -23
    assert np.all(us * 2 ** 23 == np.floor(us * 2 ** 23))   # on the 2^-23 grid
    # roughly uniform: mean and variance of U(0,1) within 5 sigma
    assert abs(us.mean() - 0.5) < 5 * math.sqrt(1 / 12 / us.size)
    assert abs(us.var() - 1 / 12) < 0.01


def test_golden_packed_bytes(orc):
    fx = json.load(open(os.path.join(GOLD, "quant_layout.json")))
    for case in fx["cases"]:
        x = np.array([case["row"]], np.float32)
        d, b = x.shape[1], case["bits"]
        for seed in (0, 1, 0xDEADBEEF12345678):
            pk = orc.quantize(x, None, b, seed)
            assert pk.tobytes().hex() == case["packed_hex"], case
            assert orc.codes(pk, d, b)[0].tolist() == case["codes"]
            # Eqn 5 reproduces the row exactly (integer grid points)
            np.testing.assert_array_equal(orc.dequant(pk, d, b)[0], x[0])


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_error_bound_and_code_range(orc, bits):
    X = synth.normal_matrix(200, 100, seed=3).numpy() * 3.0
    pk = orc.quantize(X, None, bits, seed=77)
    Q = orc.codes(pk, 100, bits)
    S, mn = orc.header(pk, 100, bits)
    L = 2 ** bits - 1
    assert Q.min() >= 0 and Q.max() <= L
    np.testing.assert_array_equal(mn, X.min(axis=1))
    np.testing.assert_allclose(S, (X.max(axis=1) - X.min(axis=1)) / L, rtol=2e-7)
    # the row minimum always codes to 0 (t = 0 and u < 1)
    assert np.all(Q[np.arange(200), X.argmin(axis=1)] == 0)
    # the row maximum codes to L or, in the rare case t < L by rounding, L-1
    qmax = Q[np.arange(200), X.argmax(axis=1)]
    assert np.all(qmax >= L - 1) and np.mean(qmax == L) > 0.95
    deq = orc.dequant(pk, 100, bits)
    err = np.abs(deq - X)
    bound = S[:, None] * (1 + 2.0 ** -20) + np.spacing(np.abs(X)) * 4
    assert np.all(err <= bound)


def test_constant_row_exact(orc):
    X = np.full((3, 17), -0.625, np.float32)
    for b in (2, 4, 8):
        pk = orc.quantize(X, None, b, seed=5)
        assert np.all(orc.codes(pk, 17, b) == 0)
        np.testing.assert_array_equal(orc.dequant(pk, 17, b), X)


def test_subnormal_scale_codes_as_constant(orc):
    # S = range / (2^b - 1) below the smallest normal float: every code is 0,
    # so de-quantization returns the row minimum (error < 255 * 2^-126).
    x = (np.float32(1e-40) * np.arange(16, dtype=np.float32))[None, :]
    for b in (2, 4, 8):
        S, _ = orc.header(orc.quantize(x, None, b, 1), 16, b)
        assert 0 < S[0] < np.finfo(np.float32).tiny
        pk = orc.quantize(x, None, b, 1)
        assert np.all(orc.codes(pk, 16, b) == 0)
        np.testing.assert_array_equal(orc.dequant(pk, 16, b), np.zeros_like(x))


def test_mask_rows_untouched(orc):
    X = synth.normal_matrix(50, 16, seed=1).numpy()
    mask = synth.bernoulli_mask(50, 0.4, seed=2).numpy()
    fill = np.full((50, orc.pitch(16, 4)), 0xAB, np.uint8)
    pk = orc.quantize(X, mask, 4, seed=9, out=fill.copy())
    assert np.all(pk[mask == 0] == 0xAB)
    full = orc.quantize(X, None, 4, seed=9)
    np.testing.assert_array_equal(pk[mask == 1], full[mask == 1])


def test_stochastic_rounding_probability(orc):
    # a row [0, 0.3, 3] at 2 bits has S = 1 and t = 0.3 for the middle
    # element: round_st rounds up with probability equal to the fraction.
    x = np.array([[0.0, 0.3, 3.0]], np.float32)
    T = 8192
    ups = sum(int(orc.codes(orc.quantize(x, None, 2, s), 3, 2)[0, 1]) for s in range(T))
    t = float(np.float32(0.3))
    sigma = math.sqrt(t * (1 - t) / T)
    assert abs(ups / T - t) < 5 * sigma


@pytest.mark.parametrize("bits", [2, 8])
def test_unbiased_and_variance_bounded(orc, bits):
    # Eqn 6: E[h^] = h; per element Var = S^2 p(1-p) <= S^2/4; averaged over
    # uniformly distributed fractions it is S^2/6.
    X = synth.normal_matrix(4, 64, seed=11).numpy()
    T = 4096
    acc = np.zeros_like(X, dtype=np.float64)
    acc2 = np.zeros_like(X, dtype=np.float64)
    for s in range(T):
        deq = orc.dequant(orc.quantize(X, None, bits, s * 7919 + 1), 64, bits).astype(np.float64)
        acc += deq
        acc2 += deq * deq
    mean = acc / T
    var = acc2 / T - mean ** 2
    S, _ = orc.header(orc.quantize(X, None, bits, 0), 64, bits)
    S = S.astype(np.float64)[:, None]
    assert np.all(np.abs(mean - X) <= 5 * S / (2 * math.sqrt(T)) + 2.0 ** -23 * S + 1e-7)
    assert np.all(var <= S * S / 4 * 1.1 + 1e-12)
    ratio = (var / (S * S)).mean()
    assert abs(ratio - 1 / 6) < 0.02


def test_round_to_nearest_would_be_biased(orc):
    # A planted mistake in a copy of the rule (round to nearest instead of
    # stochastic rounding) fails the unbiasedness check: for t = 0.3 the
    # expected code would be 0, not 0.3.  Guards the unbiasedness test's power.
    t = np.float32(0.3)
    rn = np.floor(t + 0.5)
    st = np.mean([np.floor(t + np.float32(orc.uniform(s, 0, 1))) for s in range(4096)])
    assert abs(rn - t) > 0.25 and abs(st - t) < 0.05


def test_mixed_layout_hand_example(orc):
    # widths 2, none, 8, 4 at d = 4: pitches 16, 0, 16, 16 -> offsets 0, 16, 16, 32, 48;
    # each row's bytes are the uniform quantizer's row at its own width
    X = np.array([[0, 1, 2, 3], [5, 5, 5, 5], [-1, 0, 1, 254], [0, 15, 5, 10]], np.float32)
    rbits = [2, 0, 8, 4]
    packed, roff = orc.quantize_mixed(X, rbits, 7)
    assert list(roff) == [0, 16, 16, 32, 48]
    for r, b in ((0, 2), (2, 8), (3, 4)):
        assert bytes(packed[roff[r]:roff[r + 1]]) == bytes(orc.quantize(X, None, b, 7)[r])
    M = orc.messages_mixed(X, packed, roff, rbits, 4)
    assert np.array_equal(M[0], [0, 1, 2, 3]) and np.array_equal(M[1], [5, 5, 5, 5])
    assert np.array_equal(M[3], [0, 15, 5, 10])  # integer steps of S = 1: exact
