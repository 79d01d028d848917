"""Mixed bit-widths per message row on the GPU vs the oracle (AdaQP Sec. 3.2 /
4.2: a bit-width per message; Sec. 5.3: widths drawn per message from
{2, 4, 8}): row offsets exact, packed bytes bit-exact, the aggregation over
the mixed buffer within 1e-4 (1 + |ref|) of the oracle on the GPU's own
packed bytes, for widths served by both kernels (d <= 128: lane groups with
a cp.async ring; 128 < d <= 256: a warp per edge with bulk copies)."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import close, gq, hub_graph, rmat_small, sparse_rows_graph

pytestmark = pytest.mark.gpu


def _widths(n, seed, central=0.4):
    """0 (full precision) with probability `central`, else 2, 4 or 8."""
    u = synth.uniform01(synth.stream_seed(seed, 0x42), torch.arange(n, dtype=torch.int64), 0).numpy()
    w = np.choose(np.minimum((u * 3 / (1 - central)).astype(np.int64), 2), [2, 4, 8]).astype(np.uint8)
    w[u >= 1 - central] = 0
    return w


@pytest.mark.parametrize("d", [16, 68, 128, 256])
def test_offsets_and_packed_bytes(orc, d):
    q = gq()
    n = 5000
    X = synth.normal_matrix(n, d, seed=d).numpy()
    rb = _widths(n, 1)
    rb[:5] = [0, 3, 32, 2, 8]  # widths other than 2, 4, 8 take no bytes
    pk, roff = q.quantize_pack_mixed(torch.from_numpy(X).cuda(), torch.from_numpy(rb).cuda(), 99)
    ref_pk, ref_roff = orc.quantize_mixed(X, rb, 99)
    assert np.array_equal(roff.cpu().numpy(), ref_roff)
    assert np.array_equal(pk.cpu().numpy()[:ref_roff[-1]], ref_pk)


def test_offsets_many_tiles_and_empty(orc):
    q = gq()
    for n in (0, 1, 4095, 4096, 4097, 70001):
        rb = _widths(n, n + 3) if n else np.zeros(0, np.uint8)
        roff = q.packed_row_offsets(torch.from_numpy(rb).cuda() if n else torch.zeros(0, dtype=torch.uint8,
                                                                                      device="cuda"), 200)
        sizes = np.array([orc.pitch(200, int(b)) if b in (2, 4, 8) else 0 for b in rb], np.int64)
        assert np.array_equal(roff.cpu().numpy(), np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64))


@pytest.mark.parametrize("graph", ["rmat", "hubs_split", "sparse_rows"])
@pytest.mark.parametrize("d", [16, 36, 64, 68, 128, 196, 256])
@pytest.mark.parametrize("transpose", [False, True])
def test_mixed_aggregation(orc, graph, d, transpose):
    q = gq()
    g = {"rmat": rmat_small, "hubs_split": hub_graph, "sparse_rows": sparse_rows_graph}[graph]()
    kw = dict(hub_threshold=48, split_edges=256) if graph == "hubs_split" else {}
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), **kw)
    X = synth.normal_matrix(g.n, d, seed=d + 1).numpy()
    rb = _widths(g.n, d)
    Xd, rbd = torch.from_numpy(X).cuda(), torch.from_numpy(rb).cuda()
    pk, roff = q.quantize_pack_mixed(Xd, rbd, 5)
    for coef in (0, 1):
        Y = q.dequant_spmm_mixed(G, Xd, pk, roff, rbd, coef=coef, transpose=transpose).cpu().numpy()
        M = orc.messages_mixed(X, pk.cpu().numpy(), roff.cpu().numpy(), rb, d)
        close(Y, orc.spmm(g.rowptr.numpy(), g.col.numpy(), coef, M, transpose=transpose),
              what=f"mixed d={d} coef={coef} T={transpose}")
    assert int(G.status.cpu()[0]) == 0


def test_uniform_widths_match_the_uniform_path(orc):
    # every row at 4 bits: the mixed path gives the uniform path's aggregation
    q = gq()
    g = rmat_small()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda())
    d = 128
    Xd = synth.normal_matrix(g.n, d, seed=3, device="cuda")
    rb = torch.full((g.n,), 4, dtype=torch.uint8, device="cuda")
    pk, roff = q.quantize_pack_mixed(Xd, rb, 11)
    pk_u = q.quantize_pack(Xd, None, 4, 11)
    assert torch.equal(pk[:pk_u.numel()].view(g.n, -1), pk_u)
    a = q.dequant_spmm_mixed(G, Xd, pk, roff, rb)
    b = q.dequant_spmm(G, Xd, pk_u, None, d, 4)
    close(a.cpu().numpy(), b.cpu().numpy())


def test_mixed_rejects_unsupported_width():
    q = gq()
    g = rmat_small()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda())
    Xd = synth.normal_matrix(g.n, 320, seed=3, device="cuda")
    rb = torch.full((g.n,), 2, dtype=torch.uint8, device="cuda")
    pk, roff = q.quantize_pack_mixed(Xd, rb, 1)
    with pytest.raises(q.GQError):
        q.dequant_spmm_mixed(G, Xd, pk, roff, rb)  # d = 320 is above 256
