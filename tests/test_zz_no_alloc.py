"""gq_dequant_spmm_noalloc: the aggregation for callers that cannot allocate
device memory where they aggregate, with its scratch in a fixed array
inside the library.  It must give the same result as gq_dequant_spmm (which
takes a caller workspace) on a graph whose heavy rows are split -- the case
that uses scratch -- on two calls in a row (the second finds the first
call's leftovers in the shared array), and must refuse a request larger
than its array.  This file is collected last on purpose."""
import ctypes

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


def test_noalloc_matches_workspace_entry_point_twice():
    q = gq()
    L = q.lib()
    f = _noalloc(L)
    g = hub_graph()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), 32, 256)   # split heavy rows: scratch in use
    d, bits = 128, 4
    X = synth.normal_matrix(g.n, d, seed=21, device="cuda")
    mask = synth.bernoulli_mask(g.n, 0.5, seed=22, device="cuda")
    pk = q.quantize_pack(X, mask, bits, 5)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for transpose in (0, 1):
        sc = G.c.tr_sched if transpose else G.c.sched
        assert sc.n_groups > 0 and L.gq_spmm_workspace_bytes(G.ref, transpose, d) > 0
        ref = q.dequant_spmm(G, X, pk, mask, d, bits, transpose=bool(transpose)).cpu().numpy()
        for _ in range(2):
            Y = torch.full((g.n, d), float("nan"), device="cuda")
            st = f(ctypes.byref(G.c), transpose, q.COEF_GCN, _p(X), d, _p(pk), _p(mask), d, bits, _p(Y), d, stream)
            assert st == 0, L.gq_status_string(st)
            torch.cuda.synchronize()
            close(Y.cpu().numpy(), ref, rtol=1e-4, what=f"noalloc transpose={transpose}")


def test_noalloc_rejects_requests_beyond_its_scratch():
    q = gq()
    L = q.lib()
    f = _noalloc(L)
    # one destination fed by 600,000 sources, cut into 256-edge tasks: at
    # d = 1024 the split partial rows need ~9.6 MB, above the 8 MiB array
    n = 600_000
    rowptr = torch.cat([torch.tensor([0]), torch.arange(n, 2 * n)]).to(torch.int32)
    col = torch.cat([torch.arange(n), torch.arange(1, n)]).to(torch.int32)
    G = q.graph_prepare(rowptr.cuda(), col.cuda(), 32, 256)
    d, bits = 1024, 8
    need = L.gq_spmm_workspace_bytes(G.ref, 0, d)
    assert need > L.gq_noalloc_scratch_bytes()
    pk = torch.zeros(n, q.packed_pitch(d, bits), dtype=torch.uint8, device="cuda")
    Y = torch.zeros(n, d, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = f(ctypes.byref(G.c), 0, q.COEF_GCN, None, d, _p(pk), None, d, bits, _p(Y), d, stream)
    assert st == 7 and b"fixed scratch" in L.gq_status_string(st)
    torch.cuda.synchronize()
    assert torch.count_nonzero(Y).item() == 0
