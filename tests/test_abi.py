"""C ABI checks that need no GPU: the library builds, loads and exports every
function include/qcf.h declares; host-side argument validation and fault
injection return errors before any launch; pure host helpers compute."""
import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qcf.h")


@pytest.fixture(scope="module")
def lib():
    from rag_kv_cache_re_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return _lib.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qcf_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    from rag_kv_cache_re_gb300 import _lib
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(qcf_[a-z0-9_]+)$", out, flags=re.M))
    declared = declared_functions()
    assert len(declared) >= 25
    missing = [f for f in declared if f not in exported]
    assert not missing, f"declared but not exported: {missing}"
    # the binding declares a prototype for every one of them
    assert set(declared) <= set(_lib.PROTOTYPES), set(declared) - set(_lib.PROTOTYPES)


def test_num_selected_and_version(lib):
    out = C.c_int(-1)
    assert lib.qcf_num_selected(5120, 1500, C.byref(out)) == 0 and out.value == 768
    assert lib.qcf_num_selected(96, 1500, C.byref(out)) == 0 and out.value == 15
    assert lib.qcf_num_selected(10, 10001, C.byref(out)) == 1
    assert b"sm_103a" in lib.qcf_version()


def test_rope_table_host_fill_matches_definition(lib):
    D, P = 16, 300
    cos = np.zeros((P, D // 2), np.float32)
    sin = np.zeros((P, D // 2), np.float32)
    assert lib.qcf_rope_table_fill_host(cos.ctypes.data_as(C.c_void_p), sin.ctypes.data_as(C.c_void_p), P, D,
                                        C.c_double(1e4)) == 0
    # omega_k = theta^(-2k/D): at p = 100, k = D/4 the angle is exactly 1 rad
    assert abs(cos[100, D // 4] - np.cos(1.0)) < 1e-7 and abs(sin[100, D // 4] - np.sin(1.0)) < 1e-7
    assert cos[0].tolist() == [1.0] * (D // 2) and sin[0].tolist() == [0.0] * (D // 2)


def test_argument_errors_are_synchronous(lib):
    from rag_kv_cache_re_gb300 import _lib
    fake = C.c_void_p(0x100000)  # aligned, never dereferenced: validation fails first
    assert lib.qcf_topn_select(None, 10, 3, fake, None) == 1
    assert lib.qcf_topn_select(fake, 10, 11, fake, None) == 2            # N > C
    assert lib.qcf_topn_select_workspace_size(16384) == 0
    need = lib.qcf_topn_select_workspace_size(131072)
    assert need >= 2 * 16384 * 4 and need % 4 == 0
    assert lib.qcf_topn_select_ws(fake, 131072, 10, fake, None, 0, None) == 1      # no scratch
    assert lib.qcf_topn_select_ws(fake, 131072, 10, fake, fake, need - 4, None) == 4
    assert lib.qcf_topn_select_ws(fake, 131072, 10, fake, C.c_void_p(0x100008), need, None) == 3
    assert lib.qcf_topn_select_ws(fake, 100, 0, fake, None, 0, None) == 0           # nothing to select
    assert lib.qcf_linear(fake, 4, 65, fake, 64, 0, fake, None, 0, None) == 2   # K % 64
    assert lib.qcf_linear(C.c_void_p(0x100004), 4, 64, fake, 64, 0, fake, None, 0, None) == 3  # misaligned
    assert b"16-byte" in lib.qcf_last_error()
    assert lib.qcf_sparse_causal_attn(fake, fake, 4, fake, fake, 8, 4, 4, 48, 1.0, fake, None, None, 0, None) == 2


@pytest.mark.parametrize("kind,expect", [(2, 4), (4, 3)])
def test_fault_injection_fails_before_launch(lib, kind, expect):
    fake = C.c_void_p(0x100000)
    assert lib.qcf_debug_set_fault(kind) == 0
    assert lib.qcf_linear(fake, 4, 64, fake, 64, 0, fake, None, 0, None) == expect
    # the fault fires once
    assert lib.qcf_debug_set_fault(0) == 0


def test_injected_bad_index_table(lib):
    fake = C.c_void_p(0x100000)
    assert lib.qcf_debug_set_fault(1) == 0
    assert lib.qcf_gather_rows(fake, 10, 8, fake, 3, fake, None) == 1
    assert b"injected" in lib.qcf_last_error()


def test_reposition_rejects_bad_segments(lib):
    from rag_kv_cache_re_gb300 import _lib
    fake = C.c_void_p(0x100000)
    table = _lib.RopeTable(0x100000, 0x100000, 100, 16)
    starts = (C.c_int32 * 3)(0, 5, 9)
    deltas = (C.c_int32 * 2)(0, 500)   # delta beyond the table
    assert lib.qcf_rope_reposition(fake, fake, 10, 2, 16, starts, deltas, 2, C.byref(table), None) == 2
    deltas = (C.c_int32 * 2)(0, 5)
    assert lib.qcf_rope_reposition(fake, fake, 10, 2, 16, starts, deltas, 2, C.byref(table), None) == 2  # 9 != 10
