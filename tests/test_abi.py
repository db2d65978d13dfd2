"""The C-ABI library builds for sm_103a, loads, and exports every function
that include/kpooldsa.h declares; host-side argument checks answer without a
GPU (no call here reaches a kernel)."""
import ctypes
import os
import re

import pytest

from pooled_key_dsa_gb300 import build as B
from pooled_key_dsa_gb300 import kpooldsa as K

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kpooldsa.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return K.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s+\**\s*([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"kpool_build", "dsa_index", "sparse_mla_fwd"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(K.EXPORTED) | {n for n in names if hasattr(lib, n)}


def test_checked_build_exports_the_same_symbols():
    """The KPOOL_CHECKED build (internal bounds checks) links and exports every declared function."""
    import ctypes as C
    L = C.CDLL(B.build(checked=True))
    for name in _declared_functions():
        assert hasattr(L, name), name
    L.kpool_strerror.restype = C.c_char_p
    assert L.kpool_strerror(K.CODES["KPOOL_ERR_CHECK"]) == b"internal bounds check failed"


def test_version_and_strerror(lib):
    assert "sm_103a" in K.version()
    for code in range(0, 9):
        assert K.strerror(code) != "unknown error"
    assert K.strerror(99) == "unknown error"


def _closed_pairs(T):
    a, b = divmod(T, 4)
    return 2 * a * (a - 1) + a * (b + 1)


def test_workspace_geometry(lib):
    p = K.make_params()
    for T in (0, 1, 512, 4096, 32768):
        o = K.workspace_offsets(p, T, 3)
        assert o.q8 == 0 and o.total == K.workspace_bytes(p, T, 3)
        for name in ("q8", "ws", "k8", "s_k", "pair_base", "sched", "scores", "total"):
            assert getattr(o, name) % 256 == 0
        assert o.ws >= T * 32 * 128 and o.scores - o.sched >= 4 * 4
        assert o.total - o.scores >= 4 * _closed_pairs(T)
    # the headline workload's score triangle: 134,209,536 pairs
    assert _closed_pairs(32768) == 134209536
    assert K.workspace_bytes(K.make_params(d_idx=96), 64, 1) == 0


def test_host_checks_reject_bad_arguments(lib):
    p = K.make_params()
    bad = K.make_params(topk=0)
    lay = K.LayoutC(1, 64, 16, 16, 16, 16, 16, 16)   # fake non-null device pointers
    vp = ctypes.c_void_p
    # invalid parameters
    assert lib.kpool_build(vp(16), vp(16), vp(16), vp(16), 1, 64, ctypes.byref(bad), vp(16), ctypes.byref(lay),
                           None) == K.CODES["KPOOL_ERR_INVALID_ARG"]
    # layout / argument mismatch
    assert lib.kpool_build(vp(16), vp(16), vp(16), vp(32), 1, 64, ctypes.byref(p), vp(16), ctypes.byref(lay),
                           None) == K.CODES["KPOOL_ERR_INVALID_ARG"]
    # misaligned gate
    assert lib.kpool_build(vp(16), vp(20), vp(16), vp(16), 1, 64, ctypes.byref(p), vp(16), ctypes.byref(lay),
                           None) == K.CODES["KPOOL_ERR_ALIGN"]
    # row width too small for topk
    assert lib.dsa_index(vp(16), vp(16), vp(16), ctypes.byref(lay), 512, ctypes.byref(p), vp(256), 1 << 30, vp(16),
                         2048, None) == K.CODES["KPOOL_ERR_SHAPE"]
    # workspace too small
    assert lib.dsa_index(vp(16), vp(16), vp(16), ctypes.byref(lay), 8, ctypes.byref(p), vp(256), 10, vp(16), 128,
                         None) == K.CODES["KPOOL_ERR_WORKSPACE"]
    # attention: too many heads, bad alignment
    assert lib.sparse_mla_fwd(vp(16), vp(16), vp(16), 128, 64, 65, 0.1, vp(16), vp(16), None,
                              None) == K.CODES["KPOOL_ERR_SHAPE"]
    assert lib.sparse_mla_fwd(vp(8), vp(16), vp(16), 128, 64, 64, 0.1, vp(16), vp(16), None,
                              None) == K.CODES["KPOOL_ERR_ALIGN"]
    assert lib.kpool_check_status(None, None) == K.CODES["KPOOL_ERR_INVALID_ARG"]


def test_host_checks_of_the_row_block_and_host_pipeline_entries(lib):
    vp = ctypes.c_void_p
    # row blocks: negative row count, misaligned q_lat, zero rows is a no-op
    assert lib.sparse_mla_fwd_rows(vp(16), vp(16), vp(16), 128, -1, 64, 64, 0.1, vp(16), vp(16), None,
                                   None) == K.CODES["KPOOL_ERR_SHAPE"]
    assert lib.sparse_mla_fwd_rows(vp(8), vp(16), vp(16), 128, 4, 64, 64, 0.1, vp(16), vp(16), None,
                                   None) == K.CODES["KPOOL_ERR_ALIGN"]
    assert lib.sparse_mla_fwd_rows(None, None, None, 128, 0, 64, 64, 0.1, None, None, None, None) == K.KPOOL_OK
    # host pipeline: fake non-null pointers; chunk counts, nulls and layout mismatches are refused before any
    # CUDA call
    p = K.make_params()
    lay = K.LayoutC(1, 64, 16, 16, 16, 16, 16, 16)
    h = K.HostIO(*([16] * 10))
    d = K.DevIO(*([16] * 11), ctypes.pointer(lay), 16, 1 << 30, 16, 2176)
    for n_chunks in (0, K.MAX_CHUNKS + 1):
        assert lib.kpool_forward_host(ctypes.byref(h), ctypes.byref(d), 1, 64, ctypes.byref(p), n_chunks, None, None,
                                      None) == K.CODES["KPOOL_ERR_SHAPE"]
    h_null = K.HostIO(*([16] * 9 + [0]))
    assert lib.kpool_forward_host(ctypes.byref(h_null), ctypes.byref(d), 1, 64, ctypes.byref(p), 4, None, None,
                                  None) == K.CODES["KPOOL_ERR_INVALID_ARG"]
    lay_other = K.LayoutC(1, 64, 16, 32, 16, 16, 16, 16)     # built on another cu_seqlens
    d_other = K.DevIO(*([16] * 11), ctypes.pointer(lay_other), 16, 1 << 30, 16, 2176)
    assert lib.kpool_forward_host(ctypes.byref(h), ctypes.byref(d_other), 1, 64, ctypes.byref(p), 4, None, None,
                                  None) == K.CODES["KPOOL_ERR_INVALID_ARG"]
    assert lib.kpool_forward_host(ctypes.byref(h), ctypes.byref(d), 1, 32, ctypes.byref(p), 4, None, None,
                                  None) == K.CODES["KPOOL_ERR_INVALID_ARG"]     # layout T differs


def test_host_checks_of_the_projection_entries(lib):
    vp = ctypes.c_void_p
    for fn in (lib.mla_absorb_q, lib.mla_v_proj):
        # unsupported widths and head counts are refused before any launch
        for dn, dv, H in ((96, 128, 64), (128, 256, 64), (128, 128, 0), (0, 64, 4)):
            assert fn(vp(16), vp(16), 64, H, dn, dv, vp(16), None, None) == K.CODES["KPOOL_ERR_SHAPE"]
        assert fn(vp(16), vp(16), -1, 64, 128, 128, vp(16), None, None) == K.CODES["KPOOL_ERR_SHAPE"]
        assert fn(None, vp(16), 64, 64, 128, 128, vp(16), None, None) == K.CODES["KPOOL_ERR_INVALID_ARG"]
        assert fn(vp(16), vp(24), 64, 64, 128, 128, vp(16), None, None) == K.CODES["KPOOL_ERR_ALIGN"]
        assert fn(None, None, 0, 64, 128, 128, None, None, None) == K.KPOOL_OK        # T = 0: nothing to do


def test_host_checks_of_the_stall_hook(lib):
    """Unknown bits of the stall mask are rejected before any device call."""
    assert lib.kpool_debug_inject_stall(4) == K.CODES["KPOOL_ERR_INVALID_ARG"]
    assert lib.kpool_debug_inject_stall(-1) == K.CODES["KPOOL_ERR_INVALID_ARG"]


def test_host_checks_of_the_cast_entry(lib):
    vp = ctypes.c_void_p
    cast = lib.kpool_cast_e4m3
    assert cast(vp(16), -1, vp(16), None) == K.CODES["KPOOL_ERR_INVALID_ARG"]
    assert cast(None, 8, vp(16), None) == K.CODES["KPOOL_ERR_INVALID_ARG"]
    assert cast(vp(16), 8, None, None) == K.CODES["KPOOL_ERR_INVALID_ARG"]
    assert cast(vp(18), 8, vp(16), None) == K.CODES["KPOOL_ERR_ALIGN"]
    assert cast(None, 0, None, None) == K.KPOOL_OK          # nothing to convert


def test_host_checks_of_the_backward_entry(lib):
    vp = ctypes.c_void_p
    ok = [vp(16)] * 3
    bwd = lib.sparse_mla_bwd
    assert bwd(*ok, 128, 64, 65, 0.1, vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), None,
               None) == K.CODES["KPOOL_ERR_SHAPE"]                         # more than 64 heads
    assert bwd(*ok, 0, 64, 64, 0.1, vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), None,
               None) == K.CODES["KPOOL_ERR_SHAPE"]                         # W < 1
    assert bwd(*ok, 128, 64, 64, 0.1, vp(16), vp(16), None, vp(16), vp(16), vp(16), None,
               None) == K.CODES["KPOOL_ERR_INVALID_ARG"]                   # dout missing
    assert bwd(*ok, 128, 64, 64, 0.1, vp(16), vp(16), vp(16), vp(8), vp(16), vp(16), None,
               None) == K.CODES["KPOOL_ERR_ALIGN"]                         # dq misaligned
    assert bwd(*ok, 128, 64, 64, float("nan"), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), None,
               None) == K.CODES["KPOOL_ERR_INVALID_ARG"]
    assert bwd(None, None, None, 128, 0, 64, 0.1, None, None, None, None, None, None, None, None) == K.KPOOL_OK
    red = lib.kpool_measure_l2_reduce
    assert red(vp(16), -1, vp(16), 4, None) == K.CODES["KPOOL_ERR_SHAPE"]
    assert red(None, 8, vp(16), 4, None) == K.CODES["KPOOL_ERR_INVALID_ARG"]
    assert red(vp(8), 8, vp(16), 4, None) == K.CODES["KPOOL_ERR_ALIGN"]
    assert red(None, 8, None, 0, None) == K.KPOOL_OK


def test_host_checks_of_the_decode_entries(lib):
    vp = ctypes.c_void_p
    p = K.make_params()
    bad = K.make_params(d_idx=64, n_idx_heads=4)
    assert lib.dsa_decode_workspace_bytes(ctypes.byref(bad), 4, 8) == 0
    assert lib.dsa_decode_workspace_bytes(ctypes.byref(p), 4, 8) >= 4 * 8 * 32 * 4
    ok = [vp(16)] * 4
    # unsupported shape, W too small or not a multiple of 4, workspace too small, B = 0 is a no-op
    assert lib.dsa_decode_index(*ok, 8, vp(16), 8, vp(16), 4, 512, ctypes.byref(bad), vp(256), 1 << 20, vp(16), 2176,
                                None, None) == K.CODES["KPOOL_ERR_SHAPE"]
    assert lib.dsa_decode_index(*ok, 8, vp(16), 8, vp(16), 4, 512, ctypes.byref(p), vp(256), 1 << 20, vp(16), 2050,
                                None, None) == K.CODES["KPOOL_ERR_SHAPE"]
    assert lib.dsa_decode_index(*ok, 8, vp(16), 8, vp(16), 4, 512, ctypes.byref(p), vp(256), 1 << 20, vp(16), 2178,
                                None, None) == K.CODES["KPOOL_ERR_SHAPE"]
    assert lib.dsa_decode_index(*ok, 8, vp(16), 8, vp(16), 4, 512, ctypes.byref(p), vp(256), 16, vp(16), 2176,
                                None, None) == K.CODES["KPOOL_ERR_WORKSPACE"]
    assert lib.dsa_decode_index(*ok, 8, vp(16), 8, vp(16), 4, 512, ctypes.byref(p), vp(256), 1 << 20, vp(8), 2176,
                                None, None) == K.CODES["KPOOL_ERR_ALIGN"]
    assert lib.dsa_decode_index(None, None, None, None, 8, None, 8, None, 0, 512, ctypes.byref(p), None, 0, None,
                                2176, None, None) == K.KPOOL_OK
    app = lib.kpool_paged_append
    assert app(*([vp(16)] * 6), 4, vp(16), 8, 8, ctypes.byref(bad), vp(16), vp(16), None, None) == \
        K.CODES["KPOOL_ERR_SHAPE"]
    assert app(*([vp(16)] * 6), 4, vp(16), 0, 8, ctypes.byref(p), vp(16), vp(16), None, None) == \
        K.CODES["KPOOL_ERR_SHAPE"]
    assert app(vp(16), vp(16), vp(16), None, vp(16), vp(16), 4, vp(16), 8, 8, ctypes.byref(p), vp(16), vp(16), None,
               None) == K.CODES["KPOOL_ERR_INVALID_ARG"]
    assert app(*([None] * 6), 0, None, 8, 8, ctypes.byref(p), None, None, None, None) == K.KPOOL_OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(K, "_lib", None)
    monkeypatch.setattr(K, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(K.KpoolUnavailable):
        K.lib()
