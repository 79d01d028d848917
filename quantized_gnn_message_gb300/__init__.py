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


class Graph_t(ctypes.Structure):
    """Mirror of the C struct gq_graph."""
    _fields_ = [
        ("n", ctypes.c_int64), ("nnz", ctypes.c_int64),
        ("rowptr", ctypes.c_void_p), ("col", ctypes.c_void_p),
        ("tr_rowptr", ctypes.c_void_p), ("tr_col", ctypes.c_void_p), ("tr_perm", ctypes.c_void_p),
        ("dinv_in", ctypes.c_void_p), ("dinv_out", ctypes.c_void_p), ("inv_in", ctypes.c_void_p),
        ("hub_rows", ctypes.c_void_p), ("tr_hub_rows", ctypes.c_void_p),
        ("n_hub", ctypes.c_int64), ("tr_n_hub", ctypes.c_int64),
        ("hub_threshold", ctypes.c_int32), ("max_deg", ctypes.c_int32),
        ("tr_max_deg", ctypes.c_int32), ("reserved", ctypes.c_int32),
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
            _lib = L
    return _lib


def _SIGNATURES(P, I64, I, U64, F, S):
    GP = ctypes.POINTER(Graph_t)
    return [
        ("gq_status_string", [I], ctypes.c_char_p),
        ("gq_version", [], I),
        ("gq_packed_pitch", [I, I], I64),
        ("gq_packed_header_offset", [I, I], I64),
        ("gq_quantize_pack", [P, I64, I, I64, P, I, U64, P, P], I),
        ("gq_dequant_unpack", [P, I64, I, I, P, P, I64, P], I),
        ("gq_graph_storage_bytes", [I64, I64], S),
        ("gq_graph_prepare_workspace_bytes", [I64, I64], S),
        ("gq_graph_prepare", [I64, I64, P, P, I, P, S, P, S, GP, P], I),
        ("gq_dequant_spmm", [GP, I, I, P, I64, P, P, I, I, P, I64, P], I),
        ("gq_edge_spmm", [GP, I, P, I, P, I64, P, P, I, I, P, I64, P], I),
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
    def n_hub(self):
        return int(self.c.n_hub)

    @property
    def tr_n_hub(self):
        return int(self.c.tr_n_hub)


def graph_prepare(rowptr: torch.Tensor, col: torch.Tensor, hub_threshold: int = 0) -> Graph:
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
    _check(L.gq_graph_prepare(n, nnz, _ptr(rowptr), _ptr(col), hub_threshold, _ptr(storage), sb, _ptr(ws), wb,
                              ctypes.byref(g), _stream()), "gq_graph_prepare")
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
    _check(lib().gq_dequant_spmm(g.ref, int(transpose), coef, _ptr(X), ldx, _ptr(packed), _ptr(mask), d, bits,
                                 _ptr(out), _rows(out), _stream()), "gq_dequant_spmm")
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
    _check(lib().gq_edge_spmm(g.ref, int(transpose), _ptr(alpha), heads, _ptr(X), ldx, _ptr(packed), _ptr(mask),
                              d, bits, _ptr(out), _rows(out), _stream()), "gq_edge_spmm")
    return out
