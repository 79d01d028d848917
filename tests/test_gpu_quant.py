"""GPU quantizer vs the oracle: packed bytes bit-exact (AdaQP Eqn 4),
de-quantized values bit-exact (Eqn 5), over widths that span one and many
chunks, ragged tails, masks and degenerate rows."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import gq

pytestmark = pytest.mark.gpu


def _run(orc, X, mask, bits, seed):
    q = gq()
    Xd = torch.from_numpy(X).cuda()
    md = None if mask is None else torch.from_numpy(mask).cuda()
    pk = q.quantize_pack(Xd, md, bits, seed).cpu().numpy()
    ref = orc.quantize(X, mask, bits, seed)
    sel = np.ones(X.shape[0], bool) if mask is None else mask.astype(bool)
    np.testing.assert_array_equal(pk[sel], ref[sel])
    return pk, sel


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("d", [1, 3, 8, 32, 47, 64, 100, 128, 256, 300, 512, 1000, 1500])
def test_quantize_bit_exact(orc, bits, d):
    n = 257
    X = synth.normal_matrix(n, d, seed=d + bits).numpy() * np.float32(1.7)
    pk, sel = _run(orc, X, None, bits, seed=0x1234_5678_9ABC_DEF0 + d)
    q = gq()
    deq = q.dequant_unpack(torch.from_numpy(pk).cuda(), d, bits).cpu().numpy()
    np.testing.assert_array_equal(deq, orc.dequant(pk, d, bits))


@pytest.mark.parametrize("bits", [2, 8])
def test_quantize_mask_and_untouched_rows(orc, bits):
    n, d = 1000, 64
    X = synth.normal_matrix(n, d, seed=5).numpy()
    mask = synth.bernoulli_mask(n, 0.3, seed=6).numpy()
    q = gq()
    out = torch.full((n, q.packed_pitch(d, bits)), 0xCD, dtype=torch.uint8, device="cuda")
    q.quantize_pack(torch.from_numpy(X).cuda(), torch.from_numpy(mask).cuda(), bits, 99, out=out)
    pk = out.cpu().numpy()
    ref = orc.quantize(X, mask, bits, 99)
    np.testing.assert_array_equal(pk[mask == 1], ref[mask == 1])
    assert np.all(pk[mask == 0] == 0xCD)


def test_quantize_degenerate_rows(orc):
    n, d = 64, 40
    X = synth.normal_matrix(n, d, seed=7).numpy()
    X[3] = 2.5                     # constant row
    X[4] = 0.0
    X[5] = -1e-30                  # tiny constant
    X[6, :] = 1e30                 # huge constant
    X[7] = np.linspace(-1e6, 1e6, d, dtype=np.float32)
    X[8] = np.float32(1e-38) * np.arange(d, dtype=np.float32)   # S subnormal: constant coding
    X[9, :] = 0.0
    X[9, 5] = np.float32(2.0 ** -120)                             # S normal, tiny range
    for bits in (2, 4, 8):
        _run(orc, X, None, bits, seed=3)


def test_quantize_strided_rows(orc):
    n, d = 300, 60
    big = synth.normal_matrix(n, 72, seed=8).numpy()
    q = gq()
    Xd = torch.from_numpy(big).cuda()[:, :d]          # ldx = 72
    pk = q.quantize_pack(Xd, None, 4, 11).cpu().numpy()
    np.testing.assert_array_equal(pk, orc.quantize(np.ascontiguousarray(big[:, :d]), None, 4, 11))


def test_quantize_empty_and_single(orc):
    q = gq()
    X = torch.zeros(0, 16, device="cuda")
    assert q.quantize_pack(X, None, 8, 0).shape == (0, q.packed_pitch(16, 8))
    _run(orc, np.array([[3.0]], np.float32), None, 2, 1)


def test_quantize_large_rows_sampled(orc):
    # A full-size launch (1M rows x 256) checked on a sample of rows: the
    # oracle quantizes only the sampled rows (mask) at their own indices.
    q = gq()
    n, d = 1 << 20, 256
    Xd = synth.normal_matrix(n, d, seed=9, device="cuda")
    pk = q.quantize_pack(Xd, None, 2, 77).cpu().numpy()
    rows = np.random.default_rng(0).choice(n, 2048, replace=False)
    m = np.zeros(n, np.uint8)
    m[rows] = 1
    ref = orc.quantize(Xd.cpu().numpy(), m, 2, 77)
    np.testing.assert_array_equal(pk[rows], ref[rows])
