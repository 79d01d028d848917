"""A stack of GCN / GraphSAGE-mean layers over one prepared graph.

Owns the per-layer device buffers (saved activations, gradients, one
shared workspace) and runs forward / backward through the C ABI layer
calls; no arithmetic happens here.  Layer l uses ReLU except the last
(AdaQP Sec. 2.1 layer form with sigma = ReLU on hidden layers).
"""
from __future__ import annotations

import torch

from . import (ACT_NONE, ACT_RELU, COEF_GCN, Graph, Workspace, gcn_layer_bwd, gcn_layer_fwd, lib)

# stages traced per call (see gq_gcn_layer_fwd / gq_gcn_layer_bwd)
FWD_STAGES = ("quantize", "aggregate", "update_gemm")
BWD_STAGES = ("dz", "dw_gemm", "da_gemm", "quantize_bwd", "aggregate_t")


def launches_fwd(bits: int) -> int:
    """Kernels one gq_gcn_layer_fwd call launches: [quantize] + aggregate
    + W transpose + GEMM."""
    return (1 if bits < 32 else 0) + 3


def launches_bwd(bits: int, need_dinput: bool, dz_given: bool = False) -> int:
    """[dZ] + weight GEMM + split reduction [+ W convert + dA GEMM +
    [quantize] + transposed aggregate]."""
    n = 2 if dz_given else 3
    if need_dinput:
        n += 3 + (1 if bits < 32 else 0)
    return n


class GCNStack:
    def __init__(self, g: Graph, widths, mask: torch.Tensor | None, coef: int = COEF_GCN,
                 device="cuda", keep_dA: bool = False, fuse_dz: bool = True):
        self.g = g
        self.widths = tuple(widths)
        self.L = len(widths) - 1
        self.mask = mask
        self.coef = coef
        n = g.n
        self.ws = Workspace(device)
        r8 = lambda x: (x + 7) // 8 * 8
        self.A = [torch.empty(n, r8(widths[l]), dtype=torch.bfloat16, device=device) for l in range(self.L)]
        self.H = [torch.empty(n, widths[l + 1], dtype=torch.float32, device=device) for l in range(self.L)]
        self.dH = [torch.empty(n, widths[l], dtype=torch.float32, device=device) for l in range(self.L)]
        self.dW = [torch.empty(widths[l], widths[l + 1], dtype=torch.float32, device=device) for l in range(self.L)]
        # the backward's dA = dZ W^T of each layer (the messages it quantizes), kept on request
        self.dA = [torch.empty(n, widths[l], dtype=torch.float32, device=device) if keep_dA else None
                   for l in range(self.L)]
        # fuse_dz: the transposed aggregation of layer l writes layer l-1's dZ
        # (bf16, ReLU gate applied) instead of an fp32 gradient, which layer
        # l-1 then takes as its dZ
        self.fuse_dz = fuse_dz
        self.dZ = [torch.empty(n, r8(widths[l + 1]), dtype=torch.bfloat16, device=device)
                   if fuse_dz and l < self.L - 1 else None for l in range(self.L)]
        # with fuse_dz: [H[l] > 0] as bits (written by layer l's forward GEMM),
        # the gate layer l+1's transposed aggregation applies to dZ[l]
        self.Rb = [torch.empty(n, (widths[l + 1] + 31) // 32, dtype=torch.int32, device=device)
                   if fuse_dz and l < self.L - 1 else None for l in range(self.L)]
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        L = lib()
        self.ws.get(max(int(L.gq_gcn_layer_workspace_bytes(g.ref, widths[l], widths[l + 1], 2))
                        for l in range(self.L)))

    def act(self, l: int) -> int:
        return ACT_RELU if l < self.L - 1 else ACT_NONE

    def forward(self, X: torch.Tensor, Ws, bits: int, seeds, events=None):
        h = X
        for l in range(self.L):
            ev = None if events is None else events[l]
            gcn_layer_fwd(self.g, h, Ws[l], self.mask, bits, seeds[l], self.act(l), coef=self.coef, ws=self.ws,
                          A_save=self.A[l], H_out=self.H[l], dev_err=self.err, events=ev, relu_bits=self.Rb[l])
            h = self.H[l]
        return h

    def backward(self, dY: torch.Tensor, Ws, bits: int, seeds, need_input_grad: bool = False, events=None):
        g = dY
        for l in reversed(range(self.L)):
            need = need_input_grad or l > 0
            ev = None if events is None else events[l]
            dz_in = self.dZ[l]                               # made by layer l+1 (fused), else None
            fuse = self.fuse_dz and l > 0                    # layer l makes layer l-1's dZ
            gcn_layer_bwd(self.g, None if dz_in is not None else g, self.A[l],
                          None if dz_in is not None else self.H[l], Ws[l], self.mask, bits, seeds[l],
                          self.act(l), need, coef=self.coef, ws=self.ws, dW=self.dW[l],
                          dH_in=self.dH[l] if need and not fuse else None,
                          dA_save=self.dA[l] if need else None, dev_err=self.err, events=ev, dZ_in=dz_in,
                          gate_in=self.Rb[l - 1] if fuse else None, dZ_prev=self.dZ[l - 1] if fuse else None)
            g = self.dH[l]
        return self.dW

    def launches(self, bits: int, need_input_grad: bool = False) -> int:
        return sum(launches_fwd(bits) + launches_bwd(bits, need_input_grad or l > 0, self.dZ[l] is not None)
                   for l in range(self.L))
