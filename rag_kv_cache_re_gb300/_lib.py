"""ctypes view of libqcf.so (the C ABI declared in include/qcf.h).

The library is loaded on first use.  There is no fallback: if libqcf.so has not
been built, every call raises QcfError.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libqcf.so")

STATUS_NAMES = {0: "QCF_OK", 1: "QCF_ERR_INVALID_ARG", 2: "QCF_ERR_SHAPE", 3: "QCF_ERR_ALIGN",
                4: "QCF_ERR_WORKSPACE", 5: "QCF_ERR_CUDA", 6: "QCF_ERR_TIMEOUT", 7: "QCF_ERR_UNSUPPORTED",
                8: "QCF_ERR_DEVICE"}
QCF_DEV_TIMEOUT = 0x1
QCF_DEV_BAD_INDEX = 0x2
QCF_EPI_STORE_BF16 = 0
QCF_EPI_ADD_F32 = 1
QCF_LINEAR_W_KN = 0x10


class QcfError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class RopeTable(C.Structure):
    _fields_ = [("cos", C.c_void_p), ("sin", C.c_void_p), ("max_pos", C.c_int), ("head_dim", C.c_int)]


class Dims(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("d_model", C.c_int), ("n_heads", C.c_int), ("n_kv_heads", C.c_int),
                ("head_dim", C.c_int), ("ffn", C.c_int), ("ffn_padded", C.c_int), ("vocab", C.c_int),
                ("eps", C.c_float), ("theta", C.c_float)]


class LayerWeights(C.Structure):
    _fields_ = [("w_qkv", C.c_void_p), ("w_o", C.c_void_p), ("w_gu", C.c_void_p), ("w_down", C.c_void_p),
                ("g_attn", C.c_void_p), ("g_mlp", C.c_void_p)]


class Model(C.Structure):
    _fields_ = [("dims", Dims), ("embed", C.c_void_p), ("lm_head", C.c_void_p), ("g_final", C.c_void_p),
                ("layers", C.POINTER(LayerWeights)), ("rope", RopeTable)]


class Request(C.Structure):
    _fields_ = [("n_chunks", C.c_int), ("chunk_len", C.POINTER(C.c_int32)),
                ("chunk_K_host", C.POINTER(C.c_void_p)), ("chunk_V_host", C.POINTER(C.c_void_p)),
                ("n_anchor", C.c_int), ("anchor_idx", C.POINTER(C.c_int32)),
                ("anchor_K_host", C.POINTER(C.c_void_p)), ("anchor_V_host", C.POINTER(C.c_void_p)),
                ("ids", C.c_void_p), ("query_len", C.c_int), ("crit_layer", C.c_int), ("ratio_bp", C.c_int),
                ("forced_sel", C.c_void_p), ("selector", C.c_int), ("layer_ratio_bp", C.POINTER(C.c_int32))]


class ChunkFile(C.Structure):
    _fields_ = [("fd", C.c_int), ("k_offset", C.c_int64), ("v_offset", C.c_int64), ("layer_stride", C.c_int64)]


class Outputs(C.Structure):
    _fields_ = [("K_layers", C.POINTER(C.c_void_p)), ("V_layers", C.POINTER(C.c_void_p)), ("sel", C.c_void_p),
                ("scores", C.c_void_p), ("q_crit", C.c_void_p), ("last_logits", C.c_void_p),
                ("first_token", C.c_void_p), ("first_token_host", C.c_void_p), ("x_rows", C.c_void_p),
                ("layer_sel", C.c_void_p)]


P, I, I64, F, D64, SZ = C.c_void_p, C.c_int, C.c_int64, C.c_float, C.c_double, C.c_size_t
PI32 = C.POINTER(C.c_int32)

# name -> (restype, argtypes)
PROTOTYPES = {
    "qcf_last_error": (C.c_char_p, []),
    "qcf_version": (C.c_char_p, []),
    "qcf_query_status": (I, [P, C.POINTER(C.c_uint32)]),
    "qcf_debug_set_fault": (I, [I]),
    "qcf_set_check": (I, [I]),
    "qcf_launch_count": (I64, []),
    "qcf_timing_enable": (I, [I]),
    "qcf_timing_read": (I, [I, C.POINTER(C.c_char_p), C.POINTER(D64), C.POINTER(I64), C.POINTER(I)]),
    "qcf_calibrate_exp2_rate": (I, [P, SZ, C.POINTER(D64), P]),
    "qcf_num_selected": (I, [I, I, C.POINTER(I)]),
    "qcf_rope_table_fill_host": (I, [P, P, I, I, D64]),
    "qcf_anchor_keynorm_topk": (I, [P, PI32, I, I, I, I, P, P, P]),
    "qcf_rope_reposition": (I, [P, P, I64, I, I, PI32, PI32, I, C.POINTER(RopeTable), P]),
    "qcf_profile_scores_workspace_size": (SZ, [I, I, I, I, I]),
    "qcf_profile_scores": (I, [P, P, I, I, I, I, I, F, P, P, SZ, P]),
    "qcf_profile_scores_noalloc": (I, [P, P, I, I, I, I, I, F, P, P]),
    "qcf_topn_select": (I, [P, I, I, P, P]),
    "qcf_topn_select_workspace_size": (SZ, [I]),
    "qcf_topn_select_ws": (I, [P, I, I, P, P, SZ, P]),
    "qcf_gather_rows": (I, [P, I64, I, P, I, P, P]),
    "qcf_scatter_kv": (I, [P, P, P, I, I, I, P, P, I, P]),
    "qcf_sparse_causal_attn_workspace_size": (SZ, [I, I, I, I, I]),
    "qcf_sparse_causal_attn": (I, [P, P, I, P, P, I, I, I, I, F, P, P, P, SZ, P]),
    "qcf_linear_workspace_size": (SZ, [I, I, I]),
    "qcf_linear": (I, [P, I, I, P, I, I, P, P, SZ, P]),
    "qcf_rmsnorm": (I, [P, I, I, P, F, P, P]),
    "qcf_layer_workspace_size": (SZ, [C.POINTER(Dims), I, I]),
    "qcf_fused_layer_forward": (I, [C.POINTER(Model), I, P, P, P, I, P, P, I, P, SZ, P]),
    "qcf_full_prefill_workspace_size": (SZ, [C.POINTER(Dims), I]),
    "qcf_full_prefill": (I, [C.POINTER(Model), P, I, C.POINTER(P), C.POINTER(P), P, P, P, SZ, P]),
    "qcf_request_workspace_size": (SZ, [C.POINTER(Dims), I, I, I, I]),
    "qcf_request_workspace_size_for": (SZ, [C.POINTER(Dims), C.POINTER(Request)]),
    "qcf_kv_deviation": (I, [P, P, P, I, P, P, I, I, I, P, P]),
    "qcf_storage_staging_bytes": (SZ, [C.POINTER(Dims), C.POINTER(Request)]),
    "qcf_request_prefill_storage": (I, [C.POINTER(Model), C.POINTER(Request), C.POINTER(ChunkFile), P, SZ,
                                        C.POINTER(Outputs), P, SZ, P, P]),
    "qcf_storage_status": (I, [C.POINTER(I)]),
    "qcf_batch_workspace_size": (SZ, [C.POINTER(Dims), C.POINTER(Request), I]),
    "qcf_batch_prefill": (I, [C.POINTER(Model), C.POINTER(Request), C.POINTER(Outputs), I, P, SZ, P, P,
                              C.POINTER(C.c_int64)]),
    "qcf_request_prefill": (I, [C.POINTER(Model), C.POINTER(Request), C.POINTER(Outputs), P, SZ, P, P]),
    "qcf_embed_rows": (I, [C.POINTER(Model), P, P, I, P, P]),
    "qcf_lm_head_workspace_size": (SZ, [C.POINTER(Dims)]),
    "qcf_lm_head": (I, [C.POINTER(Model), P, P, P, P, SZ, P]),
}

_lock = threading.Lock()
_lib = None


def lib() -> C.CDLL:
    """The loaded library (raises QcfError if it was never built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise QcfError("load", 7, f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
            h = C.CDLL(LIB_PATH, mode=C.RTLD_GLOBAL)
            for name, (res, args) in PROTOTYPES.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
    return _lib


def call(name: str, *args):
    """Calls a status-returning entry point and raises QcfError on failure."""
    st = getattr(lib(), name)(*args)
    if st != 0:
        raise QcfError(name, st, lib().qcf_last_error().decode(errors="replace"))
    return st
