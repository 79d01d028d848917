"""The layer stack the benchmark times (model.GCNStack: GCN layers with
ReLU on the hidden layers, AdaQP Sec. 2.1 / Sancus Sec. 2) end to end:
  - without quantization (bits = 32), against the oracle's layers chained on
    the oracle's own outputs (no teacher forcing): the output and every
    layer's dW within the bf16 tensor-core bar 2e-2 (1 + |ref|);
  - with quantization, statistically (AdaQP Sec. 2.3, Eqn 6): a one-layer
    stack's output is linear in the messages, so its mean over many seeds
    converges to the unquantized output (checked within 6 standard errors);
    through three layers the relative error against the unquantized output
    shrinks as the bit-width grows and is small at 8 bits."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import close, gq, hub_graph, rmat_small

pytestmark = pytest.mark.gpu


def _setup(widths, mask_frac, seed=0, n=3000):
    q = gq()
    g = rmat_small(scale=12, n=n, deg=12, seed=seed + 1)
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda())
    X = synth.normal_matrix(g.n, widths[0], seed=seed + 2)
    Ws = [synth.glorot(widths[l], widths[l + 1], seed=seed + 3 + l) for l in range(len(widths) - 1)]
    mask = synth.bernoulli_mask(g.n, mask_frac, seed=seed + 9)
    dY = synth.normal_matrix(g.n, widths[-1], seed=seed + 10, tag=synth.TAG_GRAD)
    return q, g, G, X, Ws, mask, dY


def _seeds(base, L, backward):
    return [synth.layer_seed(base, l, backward) for l in range(L)]


def test_stack_unquantized_matches_chained_oracle(orc):
    from quantized_gnn_message_gb300.model import GCNStack
    widths = (100, 128, 128, 47)
    L = len(widths) - 1
    q, g, G, X, Ws, mask, dY = _setup(widths, 0.6)
    model = GCNStack(G, widths, mask.cuda())
    Wd = [w.cuda() for w in Ws]
    out = model.forward(X.cuda(), Wd, 32, _seeds(0, L, False))
    model.backward(dY.cuda(), Wd, 32, _seeds(0, L, True), need_input_grad=True)
    torch.cuda.synchronize()
    assert int(model.err.item()) == 0 and int(G.status.cpu()[0]) == 0

    rp, co = g.rowptr.numpy(), g.col.numpy()
    mk = mask.numpy()
    H = X.numpy()
    saved = []
    for l in range(L):
        o = orc.gcn_layer_fwd(rp, co, orc.COEF_GCN, H, Ws[l].numpy(), mk, 32, 0, relu=l < L - 1)
        saved.append(o)
        H = o["H_out"].astype(np.float32)
    close(out.cpu().numpy(), saved[-1]["H_out"], rtol=2e-2, what="stack output")
    G_ = dY.numpy()
    for l in reversed(range(L)):
        o = orc.gcn_layer_bwd(rp, co, orc.COEF_GCN, G_, saved[l]["A"], saved[l]["Z"], Ws[l].numpy(), mk, 32, 0,
                              relu=l < L - 1, need_dinput=True)
        close(model.dW[l].cpu().numpy(), o["dW"], rtol=2e-2, what=f"layer {l} dW")
        G_ = o["dH_in"]
    close(model.dH[0].cpu().numpy(), G_, rtol=2e-2, what="input gradient")


def test_one_layer_stack_mean_over_seeds_is_unquantized(orc):
    from quantized_gnn_message_gb300.model import GCNStack
    widths = (64, 32)
    q, g, G, X, Ws, mask, dY = _setup(widths, 1.0)
    model = GCNStack(G, widths, mask.cuda())
    Xd, Wd = X.cuda(), [w.cuda() for w in Ws]
    ref = model.forward(Xd, Wd, 32, [0]).double().clone()
    T = 256
    s1 = torch.zeros_like(ref)
    s2 = torch.zeros_like(ref)
    for t in range(T):
        y = model.forward(Xd, Wd, 2, [synth.layer_seed(1000 + t, 0, False)]).double()
        s1 += y
        s2 += y * y
    torch.cuda.synchronize()
    mean = (s1 / T).cpu().numpy()
    var = np.maximum((s2 / T).cpu().numpy() - mean ** 2, 0.0) * T / (T - 1)
    se = np.sqrt(var / T)
    r = ref.cpu().numpy()
    # quantization noise: 6 standard errors; the bf16 store of A: 2^-8 relative
    tol = 6.0 * se + 4e-3 * (1.0 + np.abs(r))
    bad = np.abs(mean - r) > tol
    assert not bad.any(), f"{int(bad.sum())} of {bad.size} outputs biased; worst {np.abs(mean - r)[bad].max()}"
    # and the noise is really there: the seeds give different outputs
    assert float(np.median(se)) > 1e-3


def test_three_layer_stack_error_shrinks_with_bits(orc):
    from quantized_gnn_message_gb300.model import GCNStack
    widths = (100, 128, 128, 47)
    L = len(widths) - 1
    q, g, G, X, Ws, mask, dY = _setup(widths, 0.6, seed=3)
    model = GCNStack(G, widths, mask.cuda())
    Xd, Wd = X.cuda(), [w.cuda() for w in Ws]
    ref = model.forward(Xd, Wd, 32, _seeds(5, L, False)).clone()
    err = {}
    for b in (2, 4, 8):
        y = model.forward(Xd, Wd, b, _seeds(5, L, False))
        err[b] = float(torch.linalg.norm(y - ref) / torch.linalg.norm(ref))
    assert err[2] > err[4] > err[8], err
    assert err[8] < 2e-2 and err[2] < 1.0, err


# (widths, marginal fraction or None for every row packed, bits): the gated
# transposed aggregation on the warp-per-edge kernel (64 < d <= 256 with a
# mask or fp32 rows) and on the ring kernel (d <= 64, or every row packed)
FUSED_CASES = [((100, 128, 128, 47), 0.6, 2), ((64, 64, 32), 0.6, 8), ((64, 256, 32), None, 4),
               ((48, 64, 16), 0.5, 32), ((64, 200, 24), 0.3, 32)]


@pytest.mark.parametrize("widths,mask_frac,bits", FUSED_CASES)
def test_stack_fused_dz_is_bit_identical(orc, widths, mask_frac, bits):
    """The stack's fused backward (each transposed aggregation writes the
    layer below's bf16 dZ through its ReLU bits) gives exactly the weight
    gradients of the unfused one (fp32 gradient, then a separate
    gate-and-round pass)."""
    from quantized_gnn_message_gb300.model import GCNStack
    L = len(widths) - 1
    q, g, G, X, Ws, mask, dY = _setup(widths, 0.6 if mask_frac is None else mask_frac, seed=7)
    md = None if mask_frac is None else mask.cuda()
    Wd = [w.cuda() for w in Ws]
    out = []
    for fuse in (True, False):
        model = GCNStack(G, widths, md, fuse_dz=fuse)
        model.forward(X.cuda(), Wd, bits, _seeds(9, L, False))
        model.backward(dY.cuda(), Wd, bits, _seeds(9, L, True), need_input_grad=True)
        torch.cuda.synchronize()
        assert int(model.err.item()) == 0
        out.append([w.clone() for w in model.dW] + [model.dH[0].clone()])
    for a, b in zip(*out):
        assert torch.equal(a, b)


@pytest.mark.parametrize("widths,bits", [((64, 128, 128, 16), 2), ((64, 64, 16), 8)])
def test_stack_fused_dz_heavy_splits(orc, widths, bits):
    """The fused hand-off on a graph whose heavy rows are cut into several
    tasks (the gate applied where the last task of a row adds the partial
    rows), on the warp-per-edge kernel (d = 128) and the ring kernel
    (d = 64): bit-identical to the unfused stack."""
    from quantized_gnn_message_gb300.model import GCNStack
    q = gq()
    g = hub_graph()
    G = q.graph_prepare(g.rowptr.cuda(), g.col.cuda(), hub_threshold=32, split_edges=256)
    assert G.c.tr_sched.n_groups > 0 and G.c.sched.n_groups > 0
    L = len(widths) - 1
    X = synth.normal_matrix(g.n, widths[0], seed=51).cuda()
    Wd = [synth.glorot(widths[l], widths[l + 1], seed=52 + l).cuda() for l in range(L)]
    mask = synth.bernoulli_mask(g.n, 0.5, seed=55).cuda()
    dY = synth.normal_matrix(g.n, widths[-1], seed=56, tag=synth.TAG_GRAD).cuda()
    out = []
    for fuse in (True, False):
        model = GCNStack(G, widths, mask, fuse_dz=fuse)
        model.forward(X, Wd, bits, _seeds(3, L, False))
        model.backward(dY, Wd, bits, _seeds(3, L, True), need_input_grad=True)
        torch.cuda.synchronize()
        assert int(model.err.item()) == 0 and int(G.status.cpu()[0]) == 0
        out.append([w.clone() for w in model.dW] + [model.dH[0].clone()])
    for a, b in zip(*out):
        assert torch.equal(a, b)
