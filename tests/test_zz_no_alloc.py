"""gq_dequant_spmm_noalloc: the aggregation for callers that cannot allocate
device memory where they aggregate (a memory-pool hook, a plug-in that is
only lent its buffers, a path that must not block on an allocator), with its
scratch in a fixed array inside the library.  On a graph whose heavy rows
are split -- the case that uses scratch -- two calls in a row (the second
finds the first call's leftovers in the shared array) must both match the
oracle's aggregation (AdaQP Sec. 2.1 / Eqn 5; Sancus Sec. 2) within
1e-4 (1 + |ref|) and the result of gq_dequant_spmm, which takes a caller
workspace; the calls must leave the device's free memory unchanged; bad
arguments must be reported as such even where the scratch would also be
too small; and a request larger than the array must be refused.  This file
is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import close, gq, hub_graph

pytestmark = pytest.mark.gpu


def _noalloc(L):
    f = L.gq_dequant_spmm_noalloc
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [ctypes.c_void_p, I, I, P, I64, P, P, I, I, P, I64, P]
    f.restype = I
    return f


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_oracle_twice_without_allocating(orc):
    q = gq()
    L = q.lib()
    f = _noalloc(L)
    g = hub_graph()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), 32, 256)   # split heavy rows: scratch in use
    d, bits, seed = 128, 4, 5
    X = synth.normal_matrix(g.n, d, seed=21, device="cuda")
    mask = synth.bernoulli_mask(g.n, 0.5, seed=22, device="cuda")
    pk = q.quantize_pack(X, mask, bits, seed)
    Xh, mh = X.cpu().numpy(), mask.cpu().numpy()
    pk_ref = orc.quantize(Xh, mh, bits, seed)
    np.testing.assert_array_equal(pk.cpu().numpy()[mh == 1], pk_ref[mh == 1])
    M = orc.messages(Xh, pk_ref, mh, d, bits)
    rp, co = g.rowptr.numpy(), g.col.numpy()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for transpose in (0, 1):
        sc = G.c.tr_sched if transpose else G.c.sched
        assert sc.n_groups > 0 and L.gq_spmm_workspace_bytes(G.ref, transpose, d) > 0
        ref = orc.spmm(rp, co, orc.COEF_GCN, M, transpose=bool(transpose))
        ws_out = q.dequant_spmm(G, X, pk, mask, d, bits, transpose=bool(transpose)).cpu().numpy()
        Ys = [torch.full((g.n, d), float("nan"), device="cuda") for _ in range(3)]
        # a first call: the library's module (and the array) may be loaded lazily here
        assert f(ctypes.byref(G.c), transpose, q.COEF_GCN, _p(X), d, _p(pk), _p(mask), d, bits, _p(Ys[0]), d,
                 stream) == 0
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        for Y in Ys[1:]:
            st = f(ctypes.byref(G.c), transpose, q.COEF_GCN, _p(X), d, _p(pk), _p(mask), d, bits, _p(Y), d, stream)
            assert st == 0, L.gq_status_string(st)
            torch.cuda.synchronize()
            assert torch.cuda.mem_get_info()[0] == free0
            close(Y.cpu().numpy(), ref, rtol=1e-4, what=f"noalloc transpose={transpose} vs oracle")
            close(Y.cpu().numpy(), ws_out, rtol=1e-4, what=f"noalloc transpose={transpose} vs workspace call")


def _big_star():
    """One destination fed by 600,000 sources, cut into 256-edge tasks."""
    n = 600_000
    rowptr = torch.cat([torch.tensor([0]), torch.arange(n, 2 * n)]).to(torch.int32)
    col = torch.cat([torch.arange(n), torch.arange(1, n)]).to(torch.int32)
    return n, rowptr, col


def test_noalloc_rejects_requests_beyond_its_scratch():
    q = gq()
    L = q.lib()
    f = _noalloc(L)
    n, rowptr, col = _big_star()
    G = q.graph_prepare(rowptr.cuda(), col.cuda(), 32, 256)
    d, bits = 1024, 8
    need = L.gq_spmm_workspace_bytes(G.ref, 0, d)
    assert need > L.gq_noalloc_scratch_bytes()   # at d = 1024 the split partial rows need ~9.6 MB
    pk = torch.zeros(n, q.packed_pitch(d, bits), dtype=torch.uint8, device="cuda")
    Y = torch.zeros(n, d, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = f(ctypes.byref(G.c), 0, q.COEF_GCN, None, d, _p(pk), None, d, bits, _p(Y), d, stream)
    assert st == 7 and b"fixed scratch" in L.gq_status_string(st)
    # argument errors come first, also where the scratch would not suffice
    assert f(ctypes.byref(G.c), 0, q.COEF_GCN, None, d, _p(pk), None, d, 3, _p(Y), d, stream) == 1   # bits
    assert f(ctypes.byref(G.c), 0, q.COEF_GCN, None, d, None, None, d, bits, _p(Y), d, stream) == 1  # packed
    assert f(ctypes.byref(G.c), 0, q.COEF_GCN, None, 2048, _p(pk), None, 2048, bits, _p(Y), 2048,
             stream) == 2                                                                             # width
    torch.cuda.synchronize()
    assert torch.count_nonzero(Y).item() == 0
