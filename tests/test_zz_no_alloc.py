"""qcf_profile_scores_noalloc: profiling for callers that cannot allocate (GPU).

Some callers have no device allocator available when they need the scores (a
serving loop whose free memory all went to its KV-cache pool, or a fixed memory
budget that forbids cudaMalloc on the request path).  The no-allocation entry
point runs the same kernels with a fixed device array as scratch.  This test
calls it through the C ABI three times in a row, on different shapes, and
checks each result is bit for bit what qcf_profile_scores gives with a caller
workspace.  It also checks
that a shape needing more scratch than the fixed array is refused up front.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import qcfdata as qd

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, K, scale):
    nq, Hq, D = q.shape
    Cn, Hkv, _ = K.shape
    out = torch.full((Cn,), float("nan"), dtype=torch.float32, device=q.device)
    st = lib.qcf_profile_scores_noalloc(C.c_void_p(q.data_ptr()), C.c_void_p(K.data_ptr()), nq, Cn, Hq, Hkv, D,
                                        C.c_float(scale), C.c_void_p(out.data_ptr()),
                                        C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out


def _with_dirty_workspace(lib, q, K, scale):
    """qcf_profile_scores through the C ABI with a caller workspace that starts full of NaN bytes."""
    nq, Hq, D = q.shape
    Cn, Hkv, _ = K.shape
    nb = lib.qcf_profile_scores_workspace_size(nq, Cn, Hq, Hkv, D)
    ws = torch.full((max(256, nb),), 0xFF, dtype=torch.uint8, device=q.device)
    out = torch.full((Cn,), float("nan"), dtype=torch.float32, device=q.device)
    st = lib.qcf_profile_scores(C.c_void_p(q.data_ptr()), C.c_void_p(K.data_ptr()), nq, Cn, Hq, Hkv, D,
                                C.c_float(scale), C.c_void_p(out.data_ptr()), C.c_void_p(ws.data_ptr()),
                                C.c_size_t(ws.numel()), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.qcf_last_error()
    return out


def test_noalloc_matches_workspace_entry_point_bitwise():
    """Three calls in a row, the largest scratch footprint first: a later, smaller call that
    read anything the earlier call left in the shared array would differ from the
    workspace entry point, whose own workspace starts full of NaN bytes."""
    from rag_kv_cache_re_gb300 import _lib, qcf as Q
    lib = _lib.lib()
    cases = [dict(C=131072, nq=64, Hq=32, Hkv=8, D=128, scale=1.0),                 # 128k-token sweep context
             dict(C=5120, nq=64, Hq=32, Hkv=8, D=128, scale=1.0 / np.sqrt(128)),   # the 8B request's profile
             dict(C=1000, nq=8, Hq=4, Hkv=4, D=16, scale=0.25)]                     # a small ragged call
    for i, c in enumerate(cases):
        t = qd.sweep_tensors(c["C"], n_query=c["nq"], Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"], seed=100 + i, device="cuda")
        st, got = _noalloc(lib, t["Q"], t["K"], c["scale"])
        assert st == 0, lib.qcf_last_error()
        ref = _with_dirty_workspace(lib, t["Q"], t["K"], c["scale"])
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"call {i + 1}: differs from the workspace entry point"
        assert abs(got.double().sum().item() - c["Hq"] * c["nq"]) < 1e-3 * c["Hq"] * c["nq"]
    assert Q.qcf_query_status() == 0


def test_noalloc_refuses_shapes_beyond_its_scratch():
    from rag_kv_cache_re_gb300 import _lib
    lib = _lib.lib()
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    K = torch.zeros((64, 8, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(64, dtype=torch.float32, device="cuda")
    # 4M keys would need ~128 MiB of partial scores: refused before any launch (nothing is read)
    st = lib.qcf_profile_scores_noalloc(C.c_void_p(q.data_ptr()), C.c_void_p(K.data_ptr()), 64, 1 << 22, 32, 8, 128,
                                        C.c_float(1.0), C.c_void_p(out.data_ptr()), None)
    assert st == 4 and b"8388608" in lib.qcf_last_error()
