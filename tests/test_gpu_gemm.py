"""tcgen05 GEMMs vs the oracle's float64 product of the same bf16 inputs.
Bar: 2e-2 (1 + |ref|) for the bf16 tensor-core path; since both sides see
identical bf16 inputs, only fp32 accumulation order differs, and the
tests also require max error <= 1e-3 (1 + |ref|) to expose any layout or
descriptor fault, which would give O(1) errors."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import gq, close

pytestmark = pytest.mark.gpu


def _bf16(rows, cols, seed, pad=8, scale=1.0):
    q = gq()
    x = synth.normal_matrix(rows, cols, seed=seed, device="cuda") * scale
    return q.to_bf16(x, pad)


def _check(C, ref):
    close(C, ref, rtol=2e-2, what="bf16 gemm (bar)")
    close(C, ref, rtol=1e-3, what="bf16 gemm (exact inputs)")


@pytest.mark.parametrize("M", [1, 127, 128, 129, 1000, 4099])
@pytest.mark.parametrize("K,N", [(16, 16), (64, 64), (100, 47), (128, 256), (256, 256), (256, 48), (48, 128)])
def test_gemm_nt(orc, M, K, N):
    q = gq()
    A = _bf16(M, K, seed=M + K)
    B = _bf16(N, K, seed=N + 7)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for act in (q.ACT_NONE, q.ACT_RELU):
        C = q.gemm_nt(A, B, act=act, dev_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ref = orc.gemm(A.float().cpu().numpy(), B.float().cpu().numpy().T, bf16=True)
        if act == q.ACT_RELU:
            ref = np.maximum(ref, 0.0)
        _check(C.cpu().numpy(), ref)


def test_gemm_nt_large_sampled(orc):
    q = gq()
    M, K, N = 1 << 20, 256, 256
    A = _bf16(M, K, seed=1)
    B = _bf16(N, K, seed=2, scale=0.1)
    C = q.gemm_nt(A, B, act=q.ACT_RELU)
    rows = torch.from_numpy(np.random.default_rng(0).choice(M, 4096, replace=False)).cuda()
    ref = np.maximum(orc.gemm(A[rows].float().cpu().numpy(), B.float().cpu().numpy().T, bf16=True), 0)
    _check(C[rows].cpu().numpy(), ref)


@pytest.mark.parametrize("R", [1, 63, 64, 1000, 100_000])
@pytest.mark.parametrize("K1,N1", [(16, 16), (64, 64), (100, 256), (128, 47), (256, 256), (256, 48)])
def test_gemm_tn(orc, R, K1, N1):
    q = gq()
    X = _bf16(R, K1, seed=R + K1)
    Y = _bf16(R, N1, seed=R + N1 + 3)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = q.gemm_tn(X, Y, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = orc.gemm(X.float().cpu().numpy().T, Y.float().cpu().numpy(), bf16=True)
    _check(C.cpu().numpy(), ref)
    C2 = q.gemm_tn(X, Y, out=C.clone(), accumulate=True)
    _check(C2.cpu().numpy(), 2 * ref)


def test_gemm_tn_empty(orc):
    q = gq()
    X = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(0, 32, dtype=torch.bfloat16, device="cuda")
    C = q.gemm_tn(X, Y)
    assert torch.count_nonzero(C).item() == 0


def test_gemm_deterministic():
    q = gq()
    X = _bf16(200_000, 256, seed=5)
    Y = _bf16(200_000, 256, seed=6)
    assert torch.equal(q.gemm_tn(X, Y), q.gemm_tn(X, Y))


def test_to_bf16_round_nearest_even(orc):
    q = gq()
    x = torch.tensor([[1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-30, 3.0e38]], device="cuda")
    got = q.to_bf16(x).float().cpu().numpy()
    np.testing.assert_array_equal(got, orc.bf16_round(x.cpu().numpy()))


@pytest.mark.parametrize("rows,cols,lds,pad", [(1000, 47, 47, 8), (37, 1100, 1100, 8), (513, 256, 260, 8),
                                              (3, 5, 7, 1), (129, 64, 66, 16)])
def test_to_bf16_shapes(orc, rows, cols, lds, pad):
    # ragged widths, rows wider than one block pass, strided (non-vector) sources,
    # zero padding up to the padded width
    q = gq()
    base = synth.normal_matrix(rows, lds, seed=rows + cols, device="cuda")
    x = base[:, :cols]
    got = q.to_bf16(x, pad)
    dcols = (cols + pad - 1) // pad * pad
    full = got.as_strided((rows, dcols), (dcols, 1)).float().cpu().numpy()
    ref = np.zeros((rows, dcols), np.float32)
    ref[:, :cols] = orc.bf16_round(x.cpu().numpy())
    np.testing.assert_array_equal(full, ref)
