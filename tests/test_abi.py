"""Host-side checks of the C ABI: the library builds, loads, and exports every
symbol the header declares; argument errors come back before any launch (no
GPU needed for those)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "coli_moe.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(coli_moe_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._builder().build()
    return ctypes.CDLL(path)


def test_header_declares_entry_points():
    names = _declared()
    assert "coli_moe_layer_forward" in names and "coli_moe_configure" in names
    assert len(names) >= 15


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_lists_every_declared_symbol():
    import int4_routed_expert_f32_gb300 as coli
    assert sorted(coli.EXPORTS) == _declared()


def test_shape_validation_without_gpu(lib):
    import int4_routed_expert_f32_gb300 as coli
    bad = [
        (255, 128, 8, 2, 2.5, 4),     # hidden not a multiple of 128
        (256, 100, 8, 2, 2.5, 4),     # ffn not a multiple of 32
        (256, 144, 8, 2, 2.5, 4),     # ffn a multiple of 16 but not of 32
        (256, 128, 300, 2, 2.5, 4),   # too many experts
        (256, 128, 8, 9, 2.5, 4),     # top_k > n_experts
        (256, 128, 8, 2, 0.0, 4),     # routed_scale must be > 0
        (256, 128, 8, 2, 2.5, 0),     # max_tok >= 1
        (16512, 128, 8, 2, 2.5, 4),   # hidden above 16384
        (256, 16512, 8, 2, 2.5, 4),   # ffn above 16384
        (256, 128, 0, 1, 2.5, 4),     # no experts
        (256, 128, 32, 17, 2.5, 4),   # top_k above 16
        (256, 128, 8, 0, 2.5, 4),     # top_k >= 1
        (256, 128, 8, 2, 2.5, 65537), # max_tok above 65536
        (256, 128, 8, 2, float("nan"), 4),
        (256, 128, 8, 2, float("inf"), 4),
        (256, 128, 8, 2, -2.5, 4),
    ]
    for s in bad:
        with pytest.raises(coli.ColiError) as ei:
            coli.configure(*s)
        assert ei.value.code == coli.E_INVAL


def test_calls_before_configure_report_noshape(lib):
    import int4_routed_expert_f32_gb300 as coli
    coli.release()
    L = coli.lib()
    assert L.coli_moe_layer_forward(None, 1, None, None, None, None, None, None, None, None) == coli.E_NOSHAPE
    assert L.coli_moe_dbg_route(None, 1, None, None, None, None, None, None) == coli.E_NOSHAPE
    assert L.coli_moe_pack_int4(None, 4, 33, None, None, None) == coli.E_INVAL
    assert L.coli_moe_dbg_quantize(None, 31, None, None, None) == coli.E_INVAL
    assert L.coli_moe_set_path(7, 0) == coli.E_INVAL
    assert L.coli_moe_strerror(coli.E_NOSHAPE) == b"layer shape not configured"
    assert L.coli_moe_dbg_check_guards(None) == coli.E_NOSHAPE
    assert L.coli_moe_dbg_inject(coli.INJECT_GUARD, 0) == coli.E_NOSHAPE


def test_injection_kinds_are_checked(lib):
    import int4_routed_expert_f32_gb300 as coli
    L = coli.lib()
    assert L.coli_moe_dbg_inject(99, 0) == coli.E_INVAL
    assert L.coli_moe_dbg_inject(coli.INJECT_LAUNCH_FAIL, -1) == coli.E_INVAL
    assert L.coli_moe_dbg_inject(coli.INJECT_NONE, 0) == coli.OK


def test_stream_read_argument_checks(lib):
    """The bare-read reference rejects unaligned buffers, sizes that are not a
    multiple of 16, unaligned result pointers and out-of-range ring shapes
    before touching the device."""
    import int4_routed_expert_f32_gb300 as coli
    L = coli.lib()
    a, sink = 1 << 20, 1 << 21          # never dereferenced: rejected first
    assert L.coli_moe_dbg_stream_read(None, 16, 0, 0, 0, sink, None) == coli.E_INVAL
    assert L.coli_moe_dbg_stream_read(a + 8, 16, 0, 0, 0, sink, None) == coli.E_INVAL
    assert L.coli_moe_dbg_stream_read(a, 24, 0, 0, 0, sink, None) == coli.E_INVAL
    assert L.coli_moe_dbg_stream_read(a, 16, 0, 0, 0, sink + 4, None) == coli.E_INVAL
    assert L.coli_moe_dbg_stream_read(a, 16, 0, 0, 0, None, None) == coli.E_INVAL
    assert L.coli_moe_dbg_stream_read(a, 16, 1000, 0, 0, sink, None) == coli.E_INVAL    # not 1 KB steps
    assert L.coli_moe_dbg_stream_read(a, 16, 0, 1, 0, sink, None) == coli.E_INVAL       # one stage
    assert L.coli_moe_dbg_stream_read(a, 16, 65536, 4, 0, sink, None) == coli.E_INVAL   # 256 KB ring
    assert L.coli_moe_dbg_stream_read(a, 16, 0, 0, -1, sink, None) == coli.E_INVAL
