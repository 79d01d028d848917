"""Python binding of libgq -- quantized message passing on one GB300.

Argument marshalling only: every computation runs in the CUDA kernels of
libgq.so (built in-tree from csrc/ by build.py).  There is no CPU fallback:
if the library is missing or no CUDA device is present, calls raise.

PyTorch is used for device memory and streams: tensors are passed by
data_ptr(), and every call runs on torch.cuda.current_stream().
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

GQ_OK = 0
COEF_GCN, COEF_SAGE, COEF_ONE = 0, 1, 2
ACT_NONE, ACT_RELU = 0, 1


class GQError(RuntimeError):
    pass


class Sched_t(ctypes.Structure):
    """Mirror of the C struct gq_sched."""
    _fields_ = [("tasks", ctypes.c_void_p), ("groups", ctypes.c_void_p), ("n_tasks", ctypes.c_int64),
                ("n_groups", ctypes.c_int64), ("n_slots", ctypes.c_int64), ("light", ctypes.c_void_p),
                ("n_light", ctypes.c_int64)]


class Graph_t(ctypes.Structure):
    """Mirror of the C struct gq_graph."""
    _fields_ = [
        ("n", ctypes.c_int64), ("nnz", ctypes.c_int64),
        ("rowptr", ctypes.c_void_p), ("col", ctypes.c_void_p),
        ("tr_rowptr", ctypes.c_void_p), ("tr_col", ctypes.c_void_p), ("tr_perm", ctypes.c_void_p),
        ("dinv_in", ctypes.c_void_p), ("dinv_out", ctypes.c_void_p), ("inv_in", ctypes.c_void_p),
        ("sched", Sched_t), ("tr_sched", Sched_t),
        ("hub_threshold", ctypes.c_int32), ("split_edges", ctypes.c_int32),
        ("max_deg", ctypes.c_int32), ("tr_max_deg", ctypes.c_int32),
        ("status", ctypes.c_void_p),
    ]


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libgq (ctypes.CDLL).  Raises if it was not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise GQError(f"libgq.so is not built ({_build.LIB}); run quantized_gnn_message_gb300.build.build()")
            L = ctypes.CDLL(_build.LIB)
            P, I64, I, U64, F = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64, ctypes.c_float)
            S = ctypes.c_size_t
            for name, args, res in _SIGNATURES(P, I64, I, U64, F, S):
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            if L.gq_graph_struct_bytes() != ctypes.sizeof(Graph_t):
                raise GQError("gq_graph layout mismatch between libgq and its Python mirror")
            _lib = L
    return _lib


def _SIGNATURES(P, I64, I, U64, F, S):
    GP = ctypes.POINTER(Graph_t)
    return [
        ("gq_status_string", [I], ctypes.c_char_p),
        ("gq_version", [], I),
        ("gq_graph_struct_bytes", [], S),
        ("gq_noalloc_scratch_bytes", [], S),
        ("gq_packed_pitch", [I, I], I64),
        ("gq_packed_header_offset", [I, I], I64),
        ("gq_quantize_pack", [P, I64, I, I64, P, I, U64, P, P], I),
        ("gq_dequant_unpack", [P, I64, I, I, P, P, I64, P], I),
        ("gq_graph_storage_bytes", [I64, I64], S),
        ("gq_graph_prepare_workspace_bytes", [I64, I64], S),
        ("gq_graph_prepare", [I64, I64, P, P, I, I, P, S, P, S, GP, P], I),
        ("gq_spmm_workspace_bytes", [GP, I, I], S),
        ("gq_dequant_spmm", [GP, I, I, P, I64, P, P, I, I, P, I64, P, S, P], I),
        ("gq_dequant_spmm_noalloc", [GP, I, I, P, I64, P, P, I, I, P, I64, P], I),
        ("gq_edge_spmm", [GP, I, P, I, P, I64, P, P, I, I, P, I64, P, S, P], I),
        ("gq_gemm_bf16_nt", [P, I64, I, I64, P, I, I64, I, P, I64, P, P], I),
        ("gq_gemm_bf16_tn_workspace_bytes", [I64, I, I], S),
        ("gq_gemm_bf16_tn", [P, I64, I, I64, P, I, I64, P, I64, I, P, S, P, P], I),
        ("gq_to_bf16", [P, I64, I, I64, P, I64, I, P], I),
        ("gq_gcn_layer_workspace_bytes", [GP, I, I, I], S),
        ("gq_edge_softmax_workspace_bytes", [GP, I], S),
        ("gq_sddmm_edge_softmax", [GP, P, P, I, F, P, P, P, S, P], I),
        ("gq_quantize_edge_values_workspace_bytes", [GP, I], S),
        ("gq_quantize_edge_values", [GP, P, I, U64, P, P, P, S, P], I),
        ("gq_dequant_edge_values", [GP, P, P, I, P, P], I),
        ("gq_edge_spmm_alpha8", [GP, P, P, I, P, I64, P, P, I, I, P, I64, P, S, P], I),
        ("gq_gat_layer_workspace_bytes", [GP, I, I, I, I, I], S),
        ("gq_gat_layer_fwd", [GP, P, I64, I, P, P, P, I, I, F, P, I, U64, I, P, P, P, P, P, P, P, P, P, S, P, P], I),
        ("gq_gat_layer_bwd", [GP, P, P, I64, P, P, P, P, P, P, P, P, P, P, I, I, I, F, P, I, U64, P, P, P, P, P, P,
                              P, S, P, P], I),
        ("gq_gcn_layer_fwd", [GP, I, P, I64, I, P, I, P, I, U64, I, P, I64, P, I64, P, I64, P, S, P, P, P], I),
        ("gq_gcn_layer_bwd",
         [GP, I, P, I64, P, I64, P, I64, P, I64, P, I, I, P, I, U64, I, I, P, P, I64, P, I64, P, I64, P, P, S, P,
          P, P], I),
        ("gq_selftest_bounded_wait", [I, I, ctypes.c_longlong, P, P], I),
        ("gq_packed_row_offsets_workspace_bytes", [I64], S),
        ("gq_packed_row_offsets", [P, I64, I, P, P, S, P], I),
        ("gq_quantize_pack_mixed", [P, I64, I, I64, P, P, U64, P, P], I),
        ("gq_dequant_spmm_mixed", [GP, I, I, P, I64, P, P, P, I, P, I64, P, S, P], I),
        ("gq_message_variance_weights_workspace_bytes", [GP], S),
        ("gq_message_variance_weights", [GP, I, P, I64, I, P, P, S, P], I),
        ("gq_quant_error_workspace_bytes", [], S),
        ("gq_assign_bits", [P, P, I64, I, ctypes.c_double, ctypes.c_double, P, P], I),
        ("gq_quant_error", [P, I64, I, I64, P, P, I, F, P, P, S, P], I),
        ("gq_bits_for_error_workspace_bytes", [], S),
        ("gq_bits_for_error", [P, I64, I, I64, P, U64, ctypes.c_double, F, P, P, P, S, P], I),
    ]


def _check(status: int, what: str):
    if status != GQ_OK:
        msg = lib().gq_status_string(status).decode()
        raise GQError(f"{what}: {msg} (status {status})")


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(t, dtype, name):
    if t is None:
        return None
    if not t.is_cuda:
        raise GQError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise GQError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _rows(t):
    """(ld) of a row-major 2-D tensor with unit column stride."""
    if t.dim() != 2 or t.stride(1) != 1:
        raise GQError("expected a 2-D row-major tensor with unit column stride")
    return t.stride(0)


def packed_pitch(d: int, bits: int) -> int:
    return int(lib().gq_packed_pitch(d, bits))


def packed_header_offset(d: int, bits: int) -> int:
    return int(lib().gq_packed_header_offset(d, bits))


# --------------------------------------------------------------------------
# quantization
# --------------------------------------------------------------------------

def quantize_pack(X: torch.Tensor, mask: torch.Tensor | None, bits: int, seed: int,
                  out: torch.Tensor | None = None) -> torch.Tensor:
    """AdaQP Eqn 4 on the rows of X selected by mask (all rows if None).
    Returns the packed buffer (n x pitch uint8)."""
    _cuda(X, torch.float32, "X")
    _cuda(mask, torch.uint8, "mask")
    n, d = X.shape
    if out is None:
        out = torch.zeros(n, packed_pitch(d, bits), dtype=torch.uint8, device=X.device)
    _check(lib().gq_quantize_pack(_ptr(X), n, d, _rows(X), _ptr(mask), bits,
                                  seed & 0xFFFFFFFFFFFFFFFF, _ptr(out), _stream()), "gq_quantize_pack")
    return out


def dequant_unpack(packed: torch.Tensor, d: int, bits: int, mask: torch.Tensor | None = None,
                   out: torch.Tensor | None = None) -> torch.Tensor:
    _cuda(packed, torch.uint8, "packed")
    n = packed.shape[0]
    if out is None:
        out = torch.zeros(n, d, dtype=torch.float32, device=packed.device)
    _check(lib().gq_dequant_unpack(_ptr(packed), n, d, bits, _ptr(mask), _ptr(out), _rows(out), _stream()),
           "gq_dequant_unpack")
    return out


# --------------------------------------------------------------------------
# graphs
# --------------------------------------------------------------------------

@dataclass
class Graph:
    """A prepared graph: the caller's CSR (by destination) plus the derived
    transpose, degree norms and hub lists held in `storage`."""
    n: int
    nnz: int
    rowptr: torch.Tensor
    col: torch.Tensor
    storage: torch.Tensor
    c: Graph_t

    @property
    def ref(self):
        return ctypes.byref(self.c)

    def _view(self, ptr_name, count, dtype):
        ptr = getattr(self.c, ptr_name)
        base = self.storage.data_ptr()
        off = ptr - base
        esz = torch.empty((), dtype=dtype).element_size()
        return self.storage[off:off + count * esz].view(dtype)

    @property
    def tr_rowptr(self):
        return self._view("tr_rowptr", self.n + 1, torch.int32)

    @property
    def tr_col(self):
        return self._view("tr_col", self.nnz, torch.int32)

    @property
    def tr_perm(self):
        return self._view("tr_perm", self.nnz, torch.int32)

    @property
    def dinv_in(self):
        return self._view("dinv_in", self.n, torch.float32)

    @property
    def dinv_out(self):
        return self._view("dinv_out", self.n, torch.float32)

    @property
    def inv_in(self):
        return self._view("inv_in", self.n, torch.float32)

    @property
    def status(self):
        """The graph's device status word (non-zero: a bounded wait inside an
        aggregation kernel gave up); a one-element int32 tensor view."""
        return self._view("status", 1, torch.int32)

    @property
    def n_tasks(self):
        return int(self.c.sched.n_tasks)

    @property
    def tr_n_tasks(self):
        return int(self.c.tr_sched.n_tasks)

    def sched_arrays(self, transpose: bool = False):
        """(tasks [n_tasks x 4], groups [n_groups x 4]) as int32 tensors."""
        sc = self.c.tr_sched if transpose else self.c.sched
        out = []
        for ptr, cnt in ((sc.tasks, sc.n_tasks), (sc.groups, sc.n_groups)):
            off = ptr - self.storage.data_ptr()
            out.append(self.storage[off:off + cnt * 16].view(torch.int32).view(-1, 4))
        return out


def graph_prepare(rowptr: torch.Tensor, col: torch.Tensor, hub_threshold: int = 0,
                  split_edges: int = 0) -> Graph:
    _cuda(rowptr, torch.int32, "rowptr")
    _cuda(col, torch.int32, "col")
    n = rowptr.numel() - 1
    nnz = col.numel()
    L = lib()
    sb = int(L.gq_graph_storage_bytes(n, nnz))
    wb = int(L.gq_graph_prepare_workspace_bytes(n, nnz))
    storage = torch.empty(sb, dtype=torch.uint8, device=rowptr.device)
    ws = torch.empty(wb, dtype=torch.uint8, device=rowptr.device)
    g = Graph_t()
    _check(L.gq_graph_prepare(n, nnz, _ptr(rowptr), _ptr(col), hub_threshold, split_edges, _ptr(storage), sb,
                              _ptr(ws), wb, ctypes.byref(g), _stream()), "gq_graph_prepare")
    del ws
    return Graph(n, nnz, rowptr, col, storage, g)


# --------------------------------------------------------------------------
# aggregation
# --------------------------------------------------------------------------

def dequant_spmm(g: Graph, X: torch.Tensor | None, packed: torch.Tensor | None, mask: torch.Tensor | None,
                 d: int, bits: int, coef: int = COEF_GCN, transpose: bool = False,
                 out: torch.Tensor | None = None) -> torch.Tensor:
    _cuda(X, torch.float32, "X")
    _cuda(packed, torch.uint8, "packed")
    _cuda(mask, torch.uint8, "mask")
    dev = g.rowptr.device
    if out is None:
        out = torch.empty(g.n, d, dtype=torch.float32, device=dev)
    ldx = _rows(X) if X is not None else d
    wb = int(lib().gq_spmm_workspace_bytes(g.ref, int(transpose), d))
    ws = torch.empty(max(wb, 1), dtype=torch.uint8, device=dev)
    _check(lib().gq_dequant_spmm(g.ref, int(transpose), coef, _ptr(X), ldx, _ptr(packed), _ptr(mask), d, bits,
                                 _ptr(out), _rows(out), _ptr(ws), wb, _stream()), "gq_dequant_spmm")
    return out


def packed_row_offsets(rbits: torch.Tensor, d: int) -> torch.Tensor:
    """Byte offsets (n+1 int64) of the rows of a mixed packed buffer whose
    row r has width rbits[r] (2, 4, 8; anything else: not packed)."""
    _cuda(rbits, torch.uint8, "rbits")
    n = rbits.numel()
    L = lib()
    roff = torch.empty(n + 1, dtype=torch.int64, device=rbits.device)
    wb = int(L.gq_packed_row_offsets_workspace_bytes(n))
    ws = torch.empty(max(wb, 8), dtype=torch.uint8, device=rbits.device)
    _check(L.gq_packed_row_offsets(_ptr(rbits), n, d, _ptr(roff), _ptr(ws), wb, _stream()), "gq_packed_row_offsets")
    return roff


def quantize_pack_mixed(X: torch.Tensor, rbits: torch.Tensor, seed: int, roff: torch.Tensor | None = None):
    """AdaQP Eqn 4 with a bit-width per row.  Returns (packed, roff)."""
    _cuda(X, torch.float32, "X")
    _cuda(rbits, torch.uint8, "rbits")
    n, d = X.shape
    if roff is None:
        roff = packed_row_offsets(rbits, d)
    total = int(roff[n].item())
    packed = torch.zeros(max(total, 16), dtype=torch.uint8, device=X.device)
    _check(lib().gq_quantize_pack_mixed(_ptr(X), n, d, _rows(X), _ptr(rbits), _ptr(roff),
                                        seed & 0xFFFFFFFFFFFFFFFF, _ptr(packed), _stream()), "gq_quantize_pack_mixed")
    return packed, roff


def dequant_spmm_mixed(g: Graph, X: torch.Tensor, packed: torch.Tensor, roff: torch.Tensor, rbits: torch.Tensor,
                       coef: int = COEF_GCN, transpose: bool = False, out: torch.Tensor | None = None) -> torch.Tensor:
    """The de-quantizing aggregation over a mixed packed buffer."""
    _cuda(X, torch.float32, "X")
    n, d = X.shape
    if out is None:
        out = torch.empty(n, d, dtype=torch.float32, device=X.device)
    L = lib()
    wb = int(L.gq_spmm_workspace_bytes(g.ref, 1 if transpose else 0, d))
    ws = torch.empty(max(wb, 256), dtype=torch.uint8, device=X.device)
    _check(L.gq_dequant_spmm_mixed(g.ref, 1 if transpose else 0, coef, _ptr(X), _rows(X), _ptr(packed), _ptr(roff),
                                   _ptr(rbits), d, _ptr(out), _rows(out), _ptr(ws), wb, _stream()),
           "gq_dequant_spmm_mixed")
    return out


def dequant_spmm_noalloc(g: Graph, X: torch.Tensor | None, packed: torch.Tensor | None,
                         mask: torch.Tensor | None, d: int, bits: int, coef: int = COEF_GCN,
                         transpose: bool = False, out: torch.Tensor | None = None) -> torch.Tensor:
    """dequant_spmm without a workspace: its scratch is the library's fixed
    array (gq_noalloc_scratch_bytes); larger needs raise GQError."""
    _cuda(X, torch.float32, "X")
    _cuda(packed, torch.uint8, "packed")
    _cuda(mask, torch.uint8, "mask")
    if out is None:
        out = torch.empty(g.n, d, dtype=torch.float32, device=g.rowptr.device)
    ldx = _rows(X) if X is not None else d
    _check(lib().gq_dequant_spmm_noalloc(g.ref, int(transpose), coef, _ptr(X), ldx, _ptr(packed), _ptr(mask), d,
                                         bits, _ptr(out), _rows(out), _stream()), "gq_dequant_spmm_noalloc")
    return out


def edge_spmm(g: Graph, alpha: torch.Tensor, X: torch.Tensor | None, packed: torch.Tensor | None,
              mask: torch.Tensor | None, d: int, bits: int = 32, transpose: bool = False,
              out: torch.Tensor | None = None) -> torch.Tensor:
    _cuda(alpha, torch.float32, "alpha")
    _cuda(X, torch.float32, "X")
    heads = alpha.shape[1]
    if out is None:
        out = torch.empty(g.n, d, dtype=torch.float32, device=alpha.device)
    ldx = _rows(X) if X is not None else d
    wb = int(lib().gq_spmm_workspace_bytes(g.ref, int(transpose), d))
    ws = torch.empty(max(wb, 1), dtype=torch.uint8, device=alpha.device)
    _check(lib().gq_edge_spmm(g.ref, int(transpose), _ptr(alpha), heads, _ptr(X), ldx, _ptr(packed), _ptr(mask),
                              d, bits, _ptr(out), _rows(out), _ptr(ws), wb, _stream()), "gq_edge_spmm")
    return out


# --------------------------------------------------------------------------
# dense GEMMs
# --------------------------------------------------------------------------

def _ld_bf16(t):
    ld = _rows(t)
    if ld % 8:
        raise GQError("bf16 operands need a leading dimension that is a multiple of 8")
    return ld


def gemm_nt(A: torch.Tensor, B: torch.Tensor, act: int = ACT_NONE, out: torch.Tensor | None = None,
            dev_err: torch.Tensor | None = None) -> torch.Tensor:
    """C = act(A @ B^T) with A [M x K] and B [N x K] bf16 (views may be
    narrower than their leading dimension)."""
    _cuda(A, torch.bfloat16, "A")
    _cuda(B, torch.bfloat16, "B")
    M, K = A.shape
    N = B.shape[0]
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32, device=A.device)
    _check(lib().gq_gemm_bf16_nt(_ptr(A), M, K, _ld_bf16(A), _ptr(B), N, _ld_bf16(B), act, _ptr(out), _rows(out),
                                 _ptr(dev_err), _stream()), "gq_gemm_bf16_nt")
    return out


def gemm_tn(X: torch.Tensor, Y: torch.Tensor, out: torch.Tensor | None = None, accumulate: bool = False,
            dev_err: torch.Tensor | None = None) -> torch.Tensor:
    """C = X^T @ Y with X [R x K1] and Y [R x N1] bf16."""
    _cuda(X, torch.bfloat16, "X")
    _cuda(Y, torch.bfloat16, "Y")
    R, K1 = X.shape
    N1 = Y.shape[1]
    if out is None:
        out = torch.zeros(K1, N1, dtype=torch.float32, device=X.device)
    wb = int(lib().gq_gemm_bf16_tn_workspace_bytes(R, K1, N1))
    ws = torch.empty(wb, dtype=torch.uint8, device=X.device)
    _check(lib().gq_gemm_bf16_tn(_ptr(X), R, K1, _ld_bf16(X), _ptr(Y), N1, _ld_bf16(Y), _ptr(out), _rows(out),
                                 int(accumulate), _ptr(ws), wb, _ptr(dev_err), _stream()), "gq_gemm_bf16_tn")
    return out


def to_bf16(src: torch.Tensor, pad_to: int = 8) -> torch.Tensor:
    """bf16 copy of a 2-D fp32 tensor, columns zero-padded to a multiple of
    `pad_to` (returned as a view of the unpadded width)."""
    _cuda(src, torch.float32, "src")
    rows, cols = src.shape
    dcols = (cols + pad_to - 1) // pad_to * pad_to
    dst = torch.empty(rows, dcols, dtype=torch.bfloat16, device=src.device)
    _check(lib().gq_to_bf16(_ptr(src), rows, cols, _rows(src), _ptr(dst), dcols, dcols, _stream()), "gq_to_bf16")
    return dst[:, :cols]


# --------------------------------------------------------------------------
# GCN / GraphSAGE-mean layer
# --------------------------------------------------------------------------

def message_variance_weights(g: Graph, X: torch.Tensor, coef: int = COEF_GCN,
                             out: torch.Tensor | None = None) -> torch.Tensor:
    """AdaQP's beta_k of every message row X[k] (gq_message_variance_weights)."""
    _cuda(X, torch.float32, "X")
    n, d = X.shape
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=X.device)
    L = lib()
    wb = int(L.gq_message_variance_weights_workspace_bytes(g.ref))
    ws = torch.empty(max(wb, 1), dtype=torch.uint8, device=X.device)
    _check(L.gq_message_variance_weights(g.ref, coef, _ptr(X), _rows(X), d, _ptr(out), _ptr(ws), wb, _stream()),
           "gq_message_variance_weights")
    return out


def quant_error(X: torch.Tensor, packed: torch.Tensor, mask: torch.Tensor | None, bits: int,
                eps: float = 5e-4) -> torch.Tensor:
    """Tango's Error_X of X against its packed rows (gq_quant_error), as a
    one-element float64 device tensor."""
    _cuda(X, torch.float32, "X")
    _cuda(packed, torch.uint8, "packed")
    n, d = X.shape
    L = lib()
    ws = torch.empty(int(L.gq_quant_error_workspace_bytes()), dtype=torch.uint8, device=X.device)
    err = torch.empty(1, dtype=torch.float64, device=X.device)
    m = None if mask is None else _cuda(mask, torch.uint8, "mask")
    _check(L.gq_quant_error(_ptr(X), n, d, _rows(X), _ptr(packed), _ptr(m), bits, eps, _ptr(err), _ptr(ws),
                            ws.numel(), _stream()), "gq_quant_error")
    return err


def assign_bits(beta: torch.Tensor, d: int, lam: float, gamma: float, mask: torch.Tensor | None = None,
                out: torch.Tensor | None = None) -> torch.Tensor:
    """Per-row widths in {2, 4, 8} (0 where mask is 0) from the variance
    weights beta: AdaQP Sec. 4.2 Problems 10-12 on one device (gq.h)."""
    _cuda(beta, torch.float32, "beta")
    _cuda(mask, torch.uint8, "mask")
    n = beta.numel()
    if out is None:
        out = torch.empty(n, dtype=torch.uint8, device=beta.device)
    beta = beta.contiguous()  # held until the call has been enqueued
    _check(lib().gq_assign_bits(_ptr(beta), _ptr(mask), n, d, float(lam), float(gamma), _ptr(out),
                                _stream()), "gq_assign_bits")
    return out


def bits_for_error(X: torch.Tensor, mask: torch.Tensor | None, seed: int, threshold: float = 0.3,
                   eps: float = 5e-4, err3: torch.Tensor | None = None) -> torch.Tensor:
    """Tango's bit-count rule (gq_bits_for_error): the fewest of 2, 4, 8 bits
    whose Error_X stays below the threshold, as a one-element int32 device
    tensor; err3 (three float64) receives Error_X at each width if given."""
    _cuda(X, torch.float32, "X")
    _cuda(mask, torch.uint8, "mask")
    _cuda(err3, torch.float64, "err3")
    n, d = X.shape
    L = lib()
    ws = torch.empty(int(L.gq_bits_for_error_workspace_bytes()), dtype=torch.uint8, device=X.device)
    bits = torch.empty(1, dtype=torch.int32, device=X.device)
    _check(L.gq_bits_for_error(_ptr(X), n, d, _rows(X), _ptr(mask), seed & 0xFFFFFFFFFFFFFFFF, float(threshold),
                               eps, _ptr(err3), _ptr(bits), _ptr(ws), ws.numel(), _stream()), "gq_bits_for_error")
    return bits


def selftest_bounded_wait(helper: int, complete: bool, limit_cycles: int, status: torch.Tensor):
    """Run the bounded-wait self-test (gq_selftest_bounded_wait) into the
    one-element int32 device tensor `status`, on the current stream."""
    _cuda(status, torch.int32, "status")
    _check(lib().gq_selftest_bounded_wait(helper, 1 if complete else 0, limit_cycles, _ptr(status), _stream()),
           "gq_selftest_bounded_wait")


class Workspace:
    """A reusable device scratch buffer that grows on demand."""

    def __init__(self, device="cuda"):
        self.device = device
        self.buf = torch.empty(0, dtype=torch.uint8, device=device)

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf


def _round8(x):
    return (x + 7) // 8 * 8


def _events(evs):
    """ctypes array of cudaEvent_t handles (or None) for the stage trace."""
    if evs is None:
        return None
    arr = (ctypes.c_void_p * len(evs))()
    for i, e in enumerate(evs):
        arr[i] = e.cuda_event
    return arr


def gcn_layer_fwd(g: Graph, H_in: torch.Tensor, W: torch.Tensor, mask, bits: int, seed: int, act: int,
                  coef: int = COEF_GCN, ws: Workspace | None = None, A_save=None, H_out=None,
                  dev_err: torch.Tensor | None = None, events=None, relu_bits: torch.Tensor | None = None):
    """Returns (A_save bf16 [n x d_in] view, H_out fp32 [n x d_out]).
    relu_bits (int32 [n x ceil(d_out / 32)] words, optional): receives
    [H_out > 0] as bits, the gate of this layer's dZ in the layer above's
    backward."""
    _cuda(H_in, torch.float32, "H_in")
    _cuda(W, torch.float32, "W")
    _cuda(relu_bits, torch.int32, "relu_bits")
    n, d_in = H_in.shape
    d_out = W.shape[1]
    dev = H_in.device
    lda = _round8(d_in)
    if A_save is None:
        A_save = torch.empty(n, lda, dtype=torch.bfloat16, device=dev)
    if H_out is None:
        H_out = torch.empty(n, d_out, dtype=torch.float32, device=dev)
    L = lib()
    wb = int(L.gq_gcn_layer_workspace_bytes(g.ref, d_in, d_out, bits))
    buf = (ws or Workspace(dev)).get(wb)
    W = W.contiguous()  # held until the call has been enqueued
    _check(L.gq_gcn_layer_fwd(g.ref, coef, _ptr(H_in), _rows(H_in), d_in, _ptr(W), d_out, _ptr(mask),
                              bits, seed & 0xFFFFFFFFFFFFFFFF, act, _ptr(A_save), _rows(A_save), _ptr(H_out),
                              _rows(H_out), _ptr(relu_bits), _rows(relu_bits) if relu_bits is not None else 0,
                              _ptr(buf), buf.numel(), _ptr(dev_err), _events(events), _stream()),
           "gq_gcn_layer_fwd")
    return A_save[:, :d_in], H_out


def gcn_layer_bwd(g: Graph, dH_out: torch.Tensor | None, A_save: torch.Tensor, H_out: torch.Tensor | None,
                  W: torch.Tensor, mask, bits: int, seed: int, act: int, need_dinput: bool = True,
                  coef: int = COEF_GCN, ws: Workspace | None = None, dW=None, dH_in=None, dA_save=None,
                  dev_err: torch.Tensor | None = None, events=None, dZ_in: torch.Tensor | None = None,
                  gate_in: torch.Tensor | None = None, dZ_prev: torch.Tensor | None = None):
    """Returns (dW [d_in x d_out], dH_in [n x d_in] or None).  dZ_in: the
    layer's bf16 dZ made by the layer above (dH_out, H_out unused); dZ_prev:
    write the layer below's bf16 dZ = dH_in * gate instead of an fp32 dH_in
    (then None is returned for dH_in), the gate being gate_in, the
    relu_bits of the layer below's forward."""
    _cuda(dH_out, torch.float32, "dH_out")
    _cuda(A_save, torch.bfloat16, "A_save")
    _cuda(dZ_in, torch.bfloat16, "dZ_in")
    _cuda(dZ_prev, torch.bfloat16, "dZ_prev")
    _cuda(gate_in, torch.int32, "gate_in")
    n = A_save.shape[0]
    d_in, d_out = W.shape
    dev = A_save.device
    if dW is None:
        dW = torch.empty(d_in, d_out, dtype=torch.float32, device=dev)
    if need_dinput and dH_in is None and dZ_prev is None:
        dH_in = torch.empty(n, d_in, dtype=torch.float32, device=dev)
    if dZ_prev is not None:
        dH_in = None
    Wc = W.contiguous()  # held until the call has been enqueued
    L = lib()
    wb = int(L.gq_gcn_layer_workspace_bytes(g.ref, d_in, d_out, bits))
    buf = (ws or Workspace(dev)).get(wb)
    _check(L.gq_gcn_layer_bwd(g.ref, coef, _ptr(dH_out), _rows(dH_out) if dH_out is not None else 0,
                              _ptr(dZ_in), _rows(dZ_in) if dZ_in is not None else 0,
                              _ptr(A_save), _rows(A_save), _ptr(H_out), _rows(H_out) if H_out is not None else 0,
                              _ptr(Wc), d_in, d_out, _ptr(mask), bits, seed & 0xFFFFFFFFFFFFFFFF, act,
                              int(need_dinput), _ptr(dW), _ptr(dH_in), _rows(dH_in) if dH_in is not None else 0,
                              _ptr(gate_in), _rows(gate_in) if gate_in is not None else 0,
                              _ptr(dZ_prev), _rows(dZ_prev) if dZ_prev is not None else 0, _ptr(dA_save),
                              _ptr(buf), buf.numel(), _ptr(dev_err), _events(events), _stream()),
           "gq_gcn_layer_bwd")
    return dW, (dH_in if need_dinput else None)


# --------------------------------------------------------------------------
# GAT
# --------------------------------------------------------------------------

def sddmm_edge_softmax(g: Graph, S: torch.Tensor, D: torch.Tensor, slope: float = 0.2, with_epre: bool = False):
    """alpha (E x heads) [, E_pre] of Tango Fig. 1a steps 3-4."""
    _cuda(S, torch.float32, "S")
    _cuda(D, torch.float32, "D")
    heads = S.shape[1]
    alpha = torch.empty(g.nnz, heads, dtype=torch.float32, device=S.device)
    Epre = torch.empty_like(alpha) if with_epre else None
    wb = int(lib().gq_edge_softmax_workspace_bytes(g.ref, heads))
    ws = torch.empty(max(wb, 1), dtype=torch.uint8, device=S.device)
    S, D = S.contiguous(), D.contiguous()  # held until the call has been enqueued
    _check(lib().gq_sddmm_edge_softmax(g.ref, _ptr(S), _ptr(D), heads, slope, _ptr(Epre),
                                       _ptr(alpha), _ptr(ws), wb, _stream()), "gq_sddmm_edge_softmax")
    return (alpha, Epre) if with_epre else alpha


ALPHA_SEED_TAG = 0x5851F42D4C957F2D  # GQ_ALPHA_SEED_TAG


def quantize_edge_values(g: Graph, alpha: torch.Tensor, seed: int):
    """8-bit codes (E x heads uint8) and {S, Z} headers (n x heads x 2 fp32)
    of the attention values, one quantized vector per destination and head
    (Tango Sec. 3.3, AdaQP Eqn 4)."""
    _cuda(alpha, torch.float32, "alpha")
    heads = alpha.shape[1]
    codes = torch.empty(g.nnz, heads, dtype=torch.uint8, device=alpha.device)
    hdr = torch.empty(g.n, heads, 2, dtype=torch.float32, device=alpha.device)
    wb = int(lib().gq_quantize_edge_values_workspace_bytes(g.ref, heads))
    ws = torch.empty(max(wb, 1), dtype=torch.uint8, device=alpha.device)
    alpha = alpha.contiguous()  # held until the call has been enqueued
    _check(lib().gq_quantize_edge_values(g.ref, _ptr(alpha), heads, seed & 0xFFFFFFFFFFFFFFFF,
                                         _ptr(codes), _ptr(hdr), _ptr(ws), wb, _stream()), "gq_quantize_edge_values")
    return codes, hdr


def dequant_edge_values(g: Graph, codes: torch.Tensor, hdr: torch.Tensor) -> torch.Tensor:
    """fmaf(q, S, Z) per edge and head (AdaQP Eqn 5), E x heads fp32."""
    _cuda(codes, torch.uint8, "codes")
    _cuda(hdr, torch.float32, "hdr")
    out = torch.empty(codes.shape, dtype=torch.float32, device=codes.device)
    _check(lib().gq_dequant_edge_values(g.ref, _ptr(codes), _ptr(hdr), codes.shape[1], _ptr(out), _stream()),
           "gq_dequant_edge_values")
    return out


def edge_spmm_alpha8(g: Graph, codes: torch.Tensor, hdr: torch.Tensor, X: torch.Tensor | None,
                     packed: torch.Tensor | None, mask: torch.Tensor | None, d: int, bits: int = 32,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """Forward multi-head SpMM whose attention weights are 8-bit codes."""
    _cuda(codes, torch.uint8, "codes")
    _cuda(hdr, torch.float32, "hdr")
    _cuda(X, torch.float32, "X")
    heads = codes.shape[1]
    if out is None:
        out = torch.empty(g.n, d, dtype=torch.float32, device=codes.device)
    ldx = _rows(X) if X is not None else d
    wb = int(lib().gq_spmm_workspace_bytes(g.ref, 0, d))
    ws = torch.empty(max(wb, 1), dtype=torch.uint8, device=codes.device)
    _check(lib().gq_edge_spmm_alpha8(g.ref, _ptr(codes), _ptr(hdr), heads, _ptr(X), ldx, _ptr(packed), _ptr(mask),
                                     d, bits, _ptr(out), _rows(out), _ptr(ws), wb, _stream()), "gq_edge_spmm_alpha8")
    return out


class GATLayer:
    """Buffers and calls of one GAT layer (heads x f, LeakyReLU slope).
    alpha_bits = 8 quantizes the attention values the SpMM reads."""

    def __init__(self, g: Graph, d_in: int, heads: int, f: int, slope: float = 0.2, bits: int = 32,
                 mask=None, device="cuda", alpha_bits: int = 32):
        self.g, self.d_in, self.heads, self.f, self.slope, self.bits, self.mask = g, d_in, heads, f, slope, bits, mask
        self.alpha_bits = alpha_bits
        d = heads * f
        n = g.n
        self.Hp = torch.empty(n, d, dtype=torch.float32, device=device)
        self.S = torch.empty(n, heads, dtype=torch.float32, device=device)
        self.D = torch.empty(n, heads, dtype=torch.float32, device=device)
        self.alpha = torch.empty(g.nnz, heads, dtype=torch.float32, device=device)
        self.packed = (torch.empty(n, packed_pitch(d, bits), dtype=torch.uint8, device=device)
                       if bits < 32 else None)
        self.out = torch.empty(n, d, dtype=torch.float32, device=device)
        self.dW = torch.empty(d_in, d, dtype=torch.float32, device=device)
        self.da_src = torch.empty(heads, f, dtype=torch.float32, device=device)
        self.da_dst = torch.empty(heads, f, dtype=torch.float32, device=device)
        self.dH = torch.empty(n, d_in, dtype=torch.float32, device=device)
        self.acode = (torch.empty(g.nnz, heads, dtype=torch.uint8, device=device) if alpha_bits == 8 else None)
        self.ahdr = (torch.empty(n, heads, 2, dtype=torch.float32, device=device) if alpha_bits == 8 else None)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws = Workspace(device)
        self.ws.get(int(lib().gq_gat_layer_workspace_bytes(g.ref, d_in, heads, f, bits, alpha_bits)))

    def forward(self, H, W, a_src, a_dst, seed: int = 0):
        buf = self.ws.buf
        _check(lib().gq_gat_layer_fwd(self.g.ref, _ptr(H), _rows(H), self.d_in, _ptr(W), _ptr(a_src), _ptr(a_dst),
                                      self.heads, self.f, self.slope, _ptr(self.mask), self.bits,
                                      seed & 0xFFFFFFFFFFFFFFFF, self.alpha_bits, _ptr(self.Hp), _ptr(self.S),
                                      _ptr(self.D), _ptr(self.alpha), _ptr(self.packed), _ptr(self.acode),
                                      _ptr(self.ahdr), _ptr(self.out), _ptr(buf), buf.numel(), _ptr(self.err),
                                      _stream()), "gq_gat_layer_fwd")
        return self.out

    def backward(self, dOut, H, W, a_src, a_dst, seed: int = 0, dEpre=None, dHp=None):
        buf = self.ws.buf
        _check(lib().gq_gat_layer_bwd(self.g.ref, _ptr(dOut), _ptr(H), _rows(H), _ptr(self.Hp), _ptr(self.S),
                                      _ptr(self.D), _ptr(self.alpha), _ptr(self.packed), _ptr(self.acode),
                                      _ptr(self.ahdr), _ptr(W), _ptr(a_src),
                                      _ptr(a_dst), self.d_in, self.heads, self.f, self.slope, _ptr(self.mask),
                                      self.bits, seed & 0xFFFFFFFFFFFFFFFF, _ptr(self.dW), _ptr(self.da_src),
                                      _ptr(self.da_dst), _ptr(self.dH), _ptr(dEpre), _ptr(dHp), _ptr(buf),
                                      buf.numel(), _ptr(self.err), _stream()), "gq_gat_layer_bwd")
        return self.dW, self.da_src, self.da_dst, self.dH
