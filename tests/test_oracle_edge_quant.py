"""Pins of the oracle's 8-bit edge-value quantizer (Tango Sec. 3.3: the
SpMM reads quantized node and edge features; each (destination, head)
segment of the attention values is one AdaQP Sec. 2.3 Eqn 4 vector) against
facts that do not come from the routine itself: a hand-worked graph, the
quantizer's error bound |alpha^ - alpha| <= S (AdaQP Sec. 2.3), its
unbiasedness over seeds (Eqn 6), and the codes it must give the segment's
minimum and constant segments."""
import numpy as np

import synth


def _hand():
    # rows by destination: v0 <- e0, e1, e2; v1 <- e3; v2 has no edges; v3 <- e4, e5
    rowptr = np.array([0, 3, 4, 4, 6], np.int32)
    alpha = np.zeros((6, 2), np.float32)
    # head 0 of v0: range 255/256, so S = 1/256 and 1/S = 256 exactly
    alpha[0:3, 0] = [0.0, 255 / 256, 129 / 512]  # codes 0, 255 and 64 + (u >= 1/2)
    alpha[0:3, 1] = np.float32(1 / 3)            # a constant segment: S = 0
    alpha[3] = [1.0, 1.0]                        # a single in-edge: softmax value 1
    alpha[4:6, 0] = [0.75, 0.25]
    alpha[4:6, 1] = [0.5, 0.5]
    return rowptr, alpha


def test_hand_example(orc):
    rowptr, alpha = _hand()
    for seed in range(8):
        codes, hdr = orc.quantize_edge_values(rowptr, alpha, seed)
        u = [orc.uniform(seed, e, 0) for e in range(6)]
        # v0, head 0: Z = 0, S = 1/256; t = alpha * 256 exactly
        assert hdr[0, 0].tolist() == [1 / 256, 0.0]
        expect0 = [0, 255, 64 + (1 if np.float32(64.5) + np.float32(u[2]) >= 65 else 0)]
        assert codes[0:3, 0].tolist() == expect0
        # v0, head 1 and v1: constant segments code as 0 with Z the value
        assert codes[0:3, 1].tolist() == [0, 0, 0] and hdr[0, 1].tolist() == [0.0, np.float32(1 / 3)]
        assert codes[3].tolist() == [0, 0] and hdr[1].tolist() == [[0.0, 1.0], [0.0, 1.0]]
        # v2 has no edges: its header is zero
        assert hdr[2].tolist() == [[0.0, 0.0], [0.0, 0.0]]
        # v3, head 0: Z = 0.25, S = 0.5/255; the minimum codes as 0, the maximum as 255
        assert hdr[3, 0, 1] == np.float32(0.25)
        assert hdr[3, 0, 0] == np.float32(0.5) / np.float32(255)
        assert codes[4, 0] == 255 and codes[5, 0] == 0
        deq = orc.dequant_edge_values(rowptr, codes, hdr)
        assert deq[0, 0] == 0.0 and deq[1, 0] == np.float32(255 / 256)
        assert deq[2, 0] in (np.float32(64 / 256), np.float32(65 / 256))
        assert np.all(deq[0:3, 1] == np.float32(1 / 3)) and np.all(deq[3] == 1.0)


def test_off_grid_code_follows_its_uniform(orc):
    # the code of the off-grid value is 64 + [64.5 + u(seed, e=2, k=0) >= 65]
    rowptr, alpha = _hand()
    ups = 0
    for seed in range(64):
        codes, _ = orc.quantize_edge_values(rowptr, alpha, seed)
        up = orc.uniform(seed, 2, 0) >= 0.5
        assert codes[2, 0] == 64 + up
        ups += up
    assert 16 < ups < 48  # both ways occur


def _softmax_alpha(orc, heads=4, seed=3):
    g = synth.rmat_graph(scale=10, n=1000, n_draws=1000 * 12, seed=seed)
    rp, co = g.rowptr.numpy(), g.col.numpy()
    S = synth.normal_matrix(g.n, heads, seed=seed + 1).numpy()
    D = synth.normal_matrix(g.n, heads, seed=seed + 2).numpy()
    alpha = orc.edge_softmax(rp, co, S, D, 0.2)[1].astype(np.float32)
    return rp, alpha


def test_error_bound_and_range(orc):
    rp, alpha = _softmax_alpha(orc)
    codes, hdr = orc.quantize_edge_values(rp, alpha, 11)
    deq = orc.dequant_edge_values(rp, codes, hdr).astype(np.float64)
    v_of_e = np.repeat(np.arange(rp.size - 1), np.diff(rp))
    S = hdr[v_of_e, :, 0].astype(np.float64)
    Z = hdr[v_of_e, :, 1].astype(np.float64)
    slack = 4 * np.finfo(np.float32).eps * np.maximum(np.abs(alpha), np.abs(deq))
    assert np.all(np.abs(deq - alpha) <= S + slack)
    assert np.all(deq >= Z - slack) and np.all(deq <= Z + 255 * S + slack)
    # the segment's minimum codes as 0, so its value is Z exactly
    for v in range(rp.size - 1):
        a, b = rp[v], rp[v + 1]
        if b > a:
            j = a + np.argmin(alpha[a:b], axis=0)
            assert np.all(codes[j, np.arange(alpha.shape[1])] == 0)
            assert np.array_equal(hdr[v, :, 1], alpha[a:b].min(axis=0))


def test_unbiased_over_seeds(orc):
    rp, alpha = _softmax_alpha(orc, heads=2, seed=5)
    T = 300
    acc = np.zeros(alpha.shape)
    for s in range(T):
        c, h = orc.quantize_edge_values(rp, alpha, 1000 + s)
        acc += orc.dequant_edge_values(rp, c, h)
    mean = acc / T
    v_of_e = np.repeat(np.arange(rp.size - 1), np.diff(rp))
    # S depends on the segment only, not on the seed
    S = orc.quantize_edge_values(rp, alpha, 0)[1][v_of_e, :, 0].astype(np.float64)
    # each draw's error lies within one step S with mean zero, so its
    # standard deviation is at most S / 2
    bound = 5 * S / (2 * np.sqrt(T)) + 1e-7
    assert np.all(np.abs(mean - alpha) <= bound)


def test_aggregation_with_quantized_alpha_is_within_the_bound(orc):
    # Sum_e alpha^[e,k] m_u differs from the exact aggregation by at most
    # Sum_e S[v,k] |m_u|, the error bound carried through the SpMM
    rp, alpha = _softmax_alpha(orc, heads=4, seed=7)
    g = synth.rmat_graph(scale=10, n=1000, n_draws=1000 * 12, seed=7)
    co = g.col.numpy()
    M = synth.normal_matrix(g.n, 64, seed=9).numpy().astype(np.float64)
    codes, hdr = orc.quantize_edge_values(rp, alpha, 2)
    deq = orc.dequant_edge_values(rp, codes, hdr)
    exact = orc.edge_spmm(rp, co, alpha, M)
    quant = orc.edge_spmm(rp, co, deq, M)
    v_of_e = np.repeat(np.arange(rp.size - 1), np.diff(rp))
    S = hdr[v_of_e, :, 0].astype(np.float64) * 1.0001 + 1e-9
    bound = orc.edge_spmm(rp, co, S, np.abs(M))
    assert np.all(np.abs(quant - exact) <= bound)
    assert np.abs(quant - exact).max() > 0


def test_gat_layer_with_quantized_alpha(orc):
    # The layer with alpha_bits = 8 aggregates with the quantized attention
    # values (within their error bound of alpha), and its backward's
    # transposed SpMM is the adjoint of that forward SpMM:
    # <G, out> = <dM, M> holds with the forward's values ahat, not with alpha.
    g = synth.rmat_graph(scale=7, n=120, n_draws=120 * 10, seed=4)
    rp, co = g.rowptr.numpy(), g.col.numpy()
    rng = np.random.default_rng(3)
    heads, F, din = 2, 4, 6
    H = rng.standard_normal((g.n, din))
    W = rng.standard_normal((din, heads * F))
    a_s, a_d = rng.standard_normal((heads, F)), rng.standard_normal((heads, F))
    G = rng.standard_normal((g.n, heads * F))
    o = orc.gat_layer_fwd(rp, co, H, W, a_s, a_d, heads, 0.2, bf16=False, seed=5, alpha_bits=8)
    codes, hdr = orc.quantize_edge_values(rp, o["alpha"].astype(np.float32), 5 ^ orc.ALPHA_SEED_TAG)
    v_of_e = np.repeat(np.arange(g.n), np.diff(rp))
    S = hdr[v_of_e, :, 0].astype(np.float64)
    assert np.all(np.abs(o["ahat"] - o["alpha"]) <= S + 1e-6)
    assert np.abs(o["ahat"] - o["alpha"]).max() > 0
    b = orc.gat_layer_bwd(rp, co, G, H, o["M"], o["Hp"], o["Epre"], o["alpha"], W, a_s, a_d, heads, 0.2,
                          bf16=False, ahat=o["ahat"])
    lhs, rhs = np.sum(G * o["out"]), np.sum(b["dM"] * o["M"])
    assert abs(lhs - rhs) <= 1e-10 * (1 + abs(lhs))
    b0 = orc.gat_layer_bwd(rp, co, G, H, o["M"], o["Hp"], o["Epre"], o["alpha"], W, a_s, a_d, heads, 0.2,
                           bf16=False)
    assert abs(np.sum(b0["dM"] * o["M"]) - lhs) > 1e-6


def test_quantized_gat_forward_is_unbiased(orc):
    # AdaQP Eqn 6 for both quantizers at once: with 2-bit messages and 8-bit
    # attention values the layer's output averaged over T seeds stays within
    # a CLT bound of the unquantized layer.  (Independence of the two noise
    # streams, which the alpha seed tag provides, is not what this checks:
    # at equal indices the shared stream would correlate too few pairs here
    # to move the mean past the bound.)
    g = synth.rmat_graph(scale=6, n=60, n_draws=60 * 6, seed=8)
    rp, co = g.rowptr.numpy(), g.col.numpy()
    rng = np.random.default_rng(1)
    heads, F, din = 2, 4, 5
    H = rng.standard_normal((g.n, din))
    W = rng.standard_normal((din, heads * F))
    a_s, a_d = rng.standard_normal((heads, F)), rng.standard_normal((heads, F))
    exact = orc.gat_layer_fwd(rp, co, H, W, a_s, a_d, heads, 0.2, bf16=False)["out"]
    T = 1024
    outs = np.stack([orc.gat_layer_fwd(rp, co, H, W, a_s, a_d, heads, 0.2, bits=2, seed=s, bf16=False,
                                       alpha_bits=8)["out"] for s in range(T)])
    sd = outs.std(axis=0)
    # plus fp32 rounding: the quantized path works on fp32 H' and alpha (a
    # one-edge row's min and max code deterministically, so they vary not at all)
    assert np.all(np.abs(outs.mean(axis=0) - exact) <= 5 * sd / np.sqrt(T) + 1e-5 * (1 + np.abs(exact)))
    assert sd.max() > 0
