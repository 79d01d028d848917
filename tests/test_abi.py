"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every symbol include/gq.h declares, and its host logic
(packed-row sizes, argument checks) agrees with the spec."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q():
    import quantized_gnn_message_gb300 as q
    from quantized_gnn_message_gb300 import build
    build.build()
    q.lib()
    return q


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"GQ_API\s+[\w\s\*]*?\b(gq_\w+)\s*\(", src))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_symbols()
    for must in ("gq_quantize_pack", "gq_dequant_spmm", "gq_graph_prepare", "gq_edge_spmm"):
        assert must in names


def test_library_exports_every_declared_symbol(q):
    L = ctypes.CDLL(q.library_path())
    missing = [s for s in declared_symbols() if not hasattr(L, s)]
    assert not missing, missing


def test_graph_struct_mirror(q):
    import ctypes as C
    assert q.lib().gq_graph_struct_bytes() == C.sizeof(q.Graph_t)
    assert C.sizeof(q.Sched_t) == 56


def test_packed_sizes_match_layout(q, orc):
    for d in (1, 2, 7, 8, 31, 32, 47, 64, 100, 128, 255, 256, 1000):
        for b in (2, 4, 8):
            assert q.packed_pitch(d, b) == orc.pitch(d, b)
            assert q.packed_header_offset(d, b) == orc.header_offset(d, b)
            assert q.packed_pitch(d, b) % 16 == 0
    assert q.packed_pitch(256, 8) == 272 and q.packed_pitch(32, 2) == 16
    assert q.packed_pitch(0, 8) == -1 and q.packed_pitch(16, 3) == -1


def test_argument_checks_without_launch(q):
    L = q.lib()
    fake = ctypes.c_void_p(0x1000)
    # bits = 3 is rejected before any CUDA call
    assert L.gq_quantize_pack(fake, 10, 16, 16, None, 3, 0, fake, None) == 1
    assert L.gq_quantize_pack(None, 10, 16, 16, None, 8, 0, fake, None) == 1
    assert L.gq_quantize_pack(fake, 10, 16, 8, None, 8, 0, fake, None) == 1          # ldx < d
    assert L.gq_quantize_pack(fake, 10, 16, 16, None, 8, 0, ctypes.c_void_p(0x1008), None) == 1  # misaligned
    assert L.gq_quantize_pack(fake, 0, 16, 16, None, 8, 0, fake, None) == 0            # empty: no-op
    assert L.gq_graph_prepare(0, 0, fake, fake, 0, 0, fake, 0, fake, 0, None, None) == 1
    assert L.gq_status_string(3) == b"graph fails CSR validation"
    assert L.gq_dequant_spmm(None, 0, 0, None, 0, None, None, 16, 8, None, 16, None, 0, None) == 1
