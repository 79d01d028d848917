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


def _declarations():
    """{name: [parameter types]} of every GQ_API function in include/*.h."""
    out = {}
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        for m in re.finditer(r"GQ_API\s+[\w\s\*]*?\b(gq_\w+)\s*\(([^)]*)\)\s*;", src):
            params = " ".join(m.group(2).split())
            out[m.group(1)] = [] if params in ("", "void") else [p.strip() for p in params.split(",")]
    return out


def _kind(c_param):
    """Size and signedness class of a C parameter declaration."""
    t = c_param.rsplit(" ", 1)[0] if " " in c_param else c_param
    t = t.replace("const ", "").strip()
    if "*" in c_param or t == "gq_stream":
        return "pointer"
    return {"int": "i32", "int32_t": "i32", "int64_t": "i64", "long long": "i64", "uint64_t": "u64",
            "size_t": "u64", "float": "f32", "double": "f64"}.get(t, t)


def test_binding_signatures_match_the_header(q):
    import ctypes as C
    decl = _declarations()
    table = {name: args for name, args, _ in
             q._SIGNATURES(C.c_void_p, C.c_int64, C.c_int, C.c_uint64, C.c_float, C.c_size_t)}
    def ctype_kind(a):
        if a in (C.c_float, C.c_double):
            return "f32" if a is C.c_float else "f64"
        if a is C.c_void_p or not hasattr(a, "_type_") or isinstance(a._type_, type):
            return "pointer"  # c_void_p, POINTER(...)
        signed = a(-1).value < 0
        return ("i" if signed else "u") + str(8 * C.sizeof(a))
    unbound = sorted(set(decl) - set(table))
    assert not unbound, f"declared but not bound: {unbound}"
    for name, args in table.items():
        assert name in decl, f"{name} is bound but not declared"
        want = [_kind(p) for p in decl[name]]
        got = [ctype_kind(a) for a in args]
        assert got == want, f"{name}: binding {got} vs header {want}"


def test_newer_entry_points_check_arguments_on_the_host(q):
    # each call below is refused (1 = GQ_ERR_INVALID_ARG) or is an empty
    # no-op (0) before any CUDA call, so it runs without a GPU
    import ctypes as C
    L = q.lib()
    fake = C.c_void_p(0x1000)
    # the width choice
    assert L.gq_assign_bits(fake, None, 0, 8, 0.5, 1.0, fake, None) == 0
    assert L.gq_assign_bits(fake, None, 10, 8, 1.5, 1.0, fake, None) == 1
    assert L.gq_assign_bits(fake, None, 10, 8, 0.5, -1.0, fake, None) == 1
    assert L.gq_assign_bits(fake, None, 10, 0, 0.5, 1.0, fake, None) == 1
    assert L.gq_assign_bits(None, None, 10, 8, 0.5, 1.0, fake, None) == 1
    # attention codes and the SpMM over them, without a graph
    assert L.gq_quantize_edge_values(None, fake, 4, 0, fake, fake, None, 0, None) == 1
    assert L.gq_dequant_edge_values(None, fake, fake, 4, fake, None) == 1
    assert L.gq_edge_spmm_alpha8(None, fake, fake, 4, fake, 64, None, None, 64, 32, fake, 64, None, 0, None) == 1
    # mixed widths: packed rows must be given and 16-byte aligned
    assert L.gq_dequant_spmm_mixed(None, 0, 0, fake, 64, None, fake, fake, 64, fake, 64, None, 0, None) == 1
    assert L.gq_dequant_spmm_mixed(None, 0, 0, fake, 64, C.c_void_p(0x1008), fake, fake, 64, fake, 64, None, 0,
                                   None) == 1
    # the GAT layer: alpha_bits other than 8 and 32, and codes without headers
    g = q.Graph_t()
    args = lambda ab, acode, ahdr: (C.byref(g), fake, 64, 64, fake, fake, fake, 4, 16, C.c_float(0.2), None, 32, 0,
                                    ab, fake, fake, fake, fake, None, acode, ahdr, fake, fake, 1 << 20, None, None)
    assert L.gq_gat_layer_fwd(*args(4, None, None)) == 1
    assert L.gq_gat_layer_fwd(*args(8, fake, None)) == 1
    assert L.gq_gat_layer_workspace_bytes(None, 64, 4, 16, 32, 8) == 0
