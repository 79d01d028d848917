"""The failure path of the bounded waits, checked without a GPU fault: a
wait on an mbarrier that nothing completes gives up after a short limit and
reports its code in a status word the host reads, through the helper of the
GEMMs and of the aggregation kernels alike; a barrier that completes leaves
the word at 0; and the context stays usable afterwards."""
import time

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import close, gq, rmat_small

pytestmark = pytest.mark.gpu

LIMIT = 20_000_000  # SM cycles: about 10 ms at 2 GHz


@pytest.mark.parametrize("helper", [0, 1])
def test_wait_that_never_completes_reports(helper):
    q = gq()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    q.selftest_bounded_wait(helper, False, LIMIT, st)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    assert int(st.item()) == 0x5354


@pytest.mark.parametrize("helper", [0, 1])
def test_wait_that_completes_stays_clean(helper):
    q = gq()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q.selftest_bounded_wait(helper, True, LIMIT, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_status_keeps_first_code_and_context_survives(orc):
    q = gq()
    st = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    q.selftest_bounded_wait(1, False, LIMIT, st)  # first writer wins: 7 stays
    torch.cuda.synchronize()
    assert int(st.item()) == 7
    # the context still runs kernels correctly after a wait gave up
    g = rmat_small()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda())
    X = synth.normal_matrix(g.n, 128, seed=4).numpy()
    Y = q.dequant_spmm(G, torch.from_numpy(X).cuda(), None, None, 128, 32).cpu().numpy()
    close(Y, orc.spmm(g.rowptr.numpy(), g.col.numpy(), 0, X.astype(np.float64)))
    assert int(G.status.cpu()[0]) == 0


def test_selftest_rejects_bad_arguments():
    q = gq()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(q.GQError):
        q.selftest_bounded_wait(2, False, LIMIT, st)
    with pytest.raises(q.GQError):
        q.selftest_bounded_wait(0, False, 10, st)
