"""Python binding of the qcf C ABI: argument marshalling only.

Each function here has the name of the C entry point it calls.  Torch provides
device memory and the current CUDA stream; every computation runs in the
library's CUDA kernels.  Workspaces are cached per device and reused; calls are
ordered on the current stream.
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

from . import _lib
from ._lib import QcfError, call

_WS: Dict[Tuple[int, str], torch.Tensor] = {}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def workspace(nbytes: int, device, tag: str = "main") -> torch.Tensor:
    """A cached uint8 device buffer of at least `nbytes` (grow only, 256-byte aligned)."""
    dev = torch.device(device)
    key = (dev.index if dev.index is not None else torch.cuda.current_device(), tag)
    buf = _WS.get(key)
    need = max(256, int(nbytes))
    if buf is None or buf.numel() < need:
        if buf is not None:
            torch.cuda.current_stream(dev).synchronize()
        buf = torch.empty(need, dtype=torch.uint8, device=dev)
        _WS[key] = buf
    return buf


def _need_cuda(*ts: torch.Tensor):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise QcfError("binding", 1, "tensors must be on a CUDA device")
        if t is not None and not t.is_contiguous():
            raise QcfError("binding", 1, "tensors must be contiguous")


def _i32(a) -> C.Array:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return (C.c_int32 * len(a))(*a.tolist())


# ------------------------------------------------------------------ library

def qcf_version() -> str:
    return _lib.lib().qcf_version().decode()


def qcf_last_error() -> str:
    return _lib.lib().qcf_last_error().decode(errors="replace")


def qcf_query_status(stream=None) -> int:
    v = C.c_uint32(0)
    call("qcf_query_status", _stream(stream), C.byref(v))
    return int(v.value)


def qcf_debug_set_fault(kind: int) -> None:
    call("qcf_debug_set_fault", int(kind))


def qcf_set_check(on: bool) -> None:
    call("qcf_set_check", 1 if on else 0)


def qcf_launch_count() -> int:
    return int(_lib.lib().qcf_launch_count())


def qcf_timing_enable(on: bool) -> None:
    call("qcf_timing_enable", 1 if on else 0)


def qcf_timing_read() -> Dict[str, Tuple[float, int]]:
    n = 32
    names = (C.c_char_p * n)()
    ms = (C.c_double * n)()
    cnt = (C.c_int64 * n)()
    k = C.c_int(0)
    call("qcf_timing_read", n, names, ms, cnt, C.byref(k))
    return {names[i].decode(): (float(ms[i]), int(cnt[i])) for i in range(k.value)}


def qcf_calibrate_exp2_rate(device=None) -> float:
    """exp2 evaluations per second of the special-function units of the device (measured)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    scratch = torch.empty(1 << 22, dtype=torch.float32, device=dev)
    rate = C.c_double(0.0)
    call("qcf_calibrate_exp2_rate", _ptr(scratch), scratch.numel() * 4, C.byref(rate), _stream(None))
    return float(rate.value)


def qcf_storage_status() -> int:
    """errno of the first failed storage read since the last call (0 when none); the copy
    stream must have run past the reads (synchronise first)."""
    v = C.c_int(0)
    call("qcf_storage_status", C.byref(v))
    return int(v.value)


def qcf_num_selected(C_len: int, ratio_bp: int) -> int:
    out = C.c_int(0)
    call("qcf_num_selected", int(C_len), int(ratio_bp), C.byref(out))
    return int(out.value)


class RopeTable:
    """Device cos/sin tables [max_pos][D/2] fp32 built in fp64 by the library on the host."""

    def __init__(self, max_pos: int, head_dim: int, theta: float, device):
        cos_h = torch.empty((max_pos, head_dim // 2), dtype=torch.float32).pin_memory()
        sin_h = torch.empty_like(cos_h).pin_memory()
        call("qcf_rope_table_fill_host", C.c_void_p(cos_h.data_ptr()), C.c_void_p(sin_h.data_ptr()), int(max_pos),
             int(head_dim), float(theta))
        self.cos = cos_h.to(device, non_blocking=False)
        self.sin = sin_h.to(device, non_blocking=False)
        self.max_pos, self.head_dim = int(max_pos), int(head_dim)
        self.struct = _lib.RopeTable(self.cos.data_ptr(), self.sin.data_ptr(), self.max_pos, self.head_dim)


# ------------------------------------------------------------------ steps

def qcf_anchor_keynorm_topk(K: torch.Tensor, chunk_start: Sequence[int], n_anchor: int,
                            want_norms: bool = False, stream=None):
    _need_cuda(K)
    C_len, Hkv, D = K.shape
    n_chunks = len(chunk_start) - 1
    idx = torch.empty((n_chunks, n_anchor), dtype=torch.int32, device=K.device)
    norms = torch.empty(C_len, dtype=torch.float32, device=K.device) if want_norms else None
    call("qcf_anchor_keynorm_topk", _ptr(K), _i32(chunk_start), n_chunks, Hkv, D, int(n_anchor), _ptr(idx),
         _ptr(norms), _stream(stream))
    return (idx, norms) if want_norms else idx


def qcf_rope_reposition(K_src: torch.Tensor, K_dst: torch.Tensor, seg_start: Sequence[int],
                        seg_delta: Sequence[int], table: RopeTable, stream=None) -> torch.Tensor:
    _need_cuda(K_src, K_dst)
    n, Hkv, D = K_src.shape
    call("qcf_rope_reposition", _ptr(K_src), _ptr(K_dst), int(n), Hkv, D, _i32(seg_start), _i32(seg_delta),
         len(seg_delta), C.byref(table.struct), _stream(stream))
    return K_dst


def qcf_profile_scores(q: torch.Tensor, K: torch.Tensor, scale: float, stream=None) -> torch.Tensor:
    _need_cuda(q, K)
    nq, Hq, D = q.shape
    C_len, Hkv, _ = K.shape
    scores = torch.empty(C_len, dtype=torch.float32, device=q.device)
    nb = _lib.lib().qcf_profile_scores_workspace_size(nq, C_len, Hq, Hkv, D)
    ws = workspace(nb, q.device)
    call("qcf_profile_scores", _ptr(q), _ptr(K), nq, C_len, Hq, Hkv, D, float(scale), _ptr(scores), _ptr(ws),
         ws.numel(), _stream(stream))
    return scores


def qcf_topn_select(scores: torch.Tensor, N: int, stream=None) -> torch.Tensor:
    _need_cuda(scores)
    sel = torch.empty(max(int(N), 1), dtype=torch.int32, device=scores.device)
    call("qcf_topn_select", _ptr(scores), scores.numel(), int(N), _ptr(sel), _stream(stream))
    return sel[:N]


def qcf_topn_select_ws(scores: torch.Tensor, N: int, ws: torch.Tensor = None, stream=None) -> torch.Tensor:
    _need_cuda(scores)
    sel = torch.empty(max(int(N), 1), dtype=torch.int32, device=scores.device)
    if ws is None:
        ws = workspace(_lib.lib().qcf_topn_select_workspace_size(scores.numel()), scores.device, "topn")
    call("qcf_topn_select_ws", _ptr(scores), scores.numel(), int(N), _ptr(sel), _ptr(ws), ws.numel(),
         _stream(stream))
    return sel[:N]


def qcf_gather_rows(src: torch.Tensor, idx: torch.Tensor, stream=None) -> torch.Tensor:
    _need_cuda(src, idx)
    rows = src.shape[0]
    width = src.numel() // max(rows, 1)
    dst = torch.empty((idx.numel(),) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    call("qcf_gather_rows", _ptr(src), rows, width, _ptr(idx), idx.numel(), _ptr(dst), _stream(stream))
    return dst


def qcf_scatter_kv(k_new, v_new, pos, K_cache, V_cache, stream=None) -> None:
    _need_cuda(k_new, v_new, pos, K_cache, V_cache)
    n, Hkv, D = k_new.shape
    call("qcf_scatter_kv", _ptr(k_new), _ptr(v_new), _ptr(pos), n, Hkv, D, _ptr(K_cache), _ptr(V_cache),
         K_cache.shape[0], _stream(stream))


def qcf_kv_deviation(k_new, v_new, pos, K_cache, V_cache, stream=None):
    """dev[i] = |k_new[i] - K_cache[pos[i]]|^2 + |v_new[i] - V_cache[pos[i]]|^2 (fp32)."""
    _need_cuda(k_new, v_new, pos, K_cache, V_cache)
    n, Hkv, D = k_new.shape
    dev = torch.empty(n, dtype=torch.float32, device=k_new.device)
    call("qcf_kv_deviation", _ptr(k_new), _ptr(v_new), _ptr(pos), n, _ptr(K_cache), _ptr(V_cache), K_cache.shape[0],
         Hkv, D, _ptr(dev), _stream(stream))
    return dev


def qcf_sparse_causal_attn(q, pos, K, V, scale: float, want_lse: bool = False, stream=None):
    _need_cuda(q, pos, K, V)
    n, Hq, D = q.shape
    T, Hkv, _ = K.shape
    o = torch.empty_like(q)
    lse = torch.empty((n, Hq), dtype=torch.float32, device=q.device) if want_lse else None
    nb = _lib.lib().qcf_sparse_causal_attn_workspace_size(n, T, Hq, Hkv, D)
    ws = workspace(nb, q.device)
    call("qcf_sparse_causal_attn", _ptr(q), _ptr(pos), n, _ptr(K), _ptr(V), T, Hq, Hkv, D, float(scale), _ptr(o),
         _ptr(lse), _ptr(ws), ws.numel(), _stream(stream))
    return (o, lse) if want_lse else o


def qcf_linear(A: torch.Tensor, W: torch.Tensor, out: Optional[torch.Tensor] = None, add: bool = False,
               w_kn: bool = False, stream=None) -> torch.Tensor:
    """out = A W^T (bf16 out), or out += A W^T for an fp32 `out` when add=True.
    With w_kn, W is stored [K][N] and out = A W."""
    _need_cuda(A, W)
    M, K = A.shape
    N = W.shape[1] if w_kn else W.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32 if add else torch.bfloat16, device=A.device)
        if add:
            out.zero_()
    nb = _lib.lib().qcf_linear_workspace_size(M, N, K)
    ws = workspace(nb, A.device)
    epi = (_lib.QCF_EPI_ADD_F32 if add else _lib.QCF_EPI_STORE_BF16) | (_lib.QCF_LINEAR_W_KN if w_kn else 0)
    call("qcf_linear", _ptr(A), M, K, _ptr(W), N, epi, _ptr(out), _ptr(ws), ws.numel(), _stream(stream))
    return out


def qcf_rmsnorm(x: torch.Tensor, g: torch.Tensor, eps: float, stream=None) -> torch.Tensor:
    _need_cuda(x, g)
    n, d = x.shape
    h = torch.empty((n, d), dtype=torch.bfloat16, device=x.device)
    call("qcf_rmsnorm", _ptr(x), n, d, _ptr(g), float(eps), _ptr(h), _stream(stream))
    return h


def qcf_fused_layer_forward(model, layer: int, x: torch.Tensor, rope_pos: torch.Tensor, cache_row: torch.Tensor,
                            K_cache: torch.Tensor, V_cache: torch.Tensor, stream=None) -> torch.Tensor:
    _need_cuda(x, rope_pos, cache_row, K_cache, V_cache)
    n = x.shape[0]
    T = K_cache.shape[0]
    nb = _lib.lib().qcf_layer_workspace_size(C.byref(model.struct.dims), n, T)
    ws = workspace(nb, x.device)
    call("qcf_fused_layer_forward", C.byref(model.struct), int(layer), _ptr(x), _ptr(rope_pos), _ptr(cache_row), n,
         _ptr(K_cache), _ptr(V_cache), T, _ptr(ws), ws.numel(), _stream(stream))
    return x


def qcf_embed_rows(model, ids: torch.Tensor, rows: Optional[torch.Tensor], n: int, stream=None) -> torch.Tensor:
    x = torch.empty((n, model.spec.d_model), dtype=torch.float32, device=ids.device)
    call("qcf_embed_rows", C.byref(model.struct), _ptr(ids), _ptr(rows), int(n), _ptr(x), _stream(stream))
    return x


def qcf_lm_head(model, x_last: torch.Tensor, stream=None):
    logits = torch.empty(model.spec.vocab, dtype=torch.float32, device=x_last.device)
    token = torch.empty(1, dtype=torch.int32, device=x_last.device)
    nb = _lib.lib().qcf_lm_head_workspace_size(C.byref(model.struct.dims))
    ws = workspace(nb, x_last.device, tag="lm")
    call("qcf_lm_head", C.byref(model.struct), _ptr(x_last), _ptr(logits), _ptr(token), _ptr(ws), ws.numel(),
         _stream(stream))
    return logits, token


def qcf_full_prefill(model, ids: torch.Tensor, K_layers: Optional[List[torch.Tensor]] = None,
                     V_layers: Optional[List[torch.Tensor]] = None, stream=None):
    """Full recompute of ids (device int32 [T]) -> per-layer K/V, last logits, first token (device)."""
    _need_cuda(ids)
    s = model.spec
    T = ids.numel()
    dev = ids.device
    if K_layers is None:
        K_layers = [torch.empty((T, s.n_kv_heads, s.head_dim), dtype=torch.bfloat16, device=dev) for _ in range(s.n_layers)]
        V_layers = [torch.empty_like(K_layers[0]) for _ in range(s.n_layers)]
    kp = (C.c_void_p * s.n_layers)(*[k.data_ptr() for k in K_layers])
    vp = (C.c_void_p * s.n_layers)(*[v.data_ptr() for v in V_layers])
    logits = torch.empty(s.vocab, dtype=torch.float32, device=dev)
    token = torch.empty(1, dtype=torch.int32, device=dev)
    nb = _lib.lib().qcf_full_prefill_workspace_size(C.byref(model.struct.dims), T)
    ws = workspace(nb, dev)
    call("qcf_full_prefill", C.byref(model.struct), _ptr(ids), T, kp, vp, _ptr(logits), _ptr(token), _ptr(ws),
         ws.numel(), _stream(stream))
    return K_layers, V_layers, logits, token


def qcf_request_prefill(model, req: "_lib.Request", outs: "_lib.Outputs", ws: torch.Tensor, compute_stream,
                        copy_stream) -> None:
    """Enqueues the fused prefill of one request (structs built by model.FusedRequest)."""
    call("qcf_request_prefill", C.byref(model.struct), C.byref(req), C.byref(outs), _ptr(ws), ws.numel(),
         C.c_void_p(compute_stream.cuda_stream), C.c_void_p(copy_stream.cuda_stream))


def qcf_batch_prefill(model, reqs, outs, ws: torch.Tensor, compute_stream, copy_stream) -> int:
    """Enqueues several fused prefills sharing their common chunks' host-to-device copies
    (structs built by model.FusedRequest); returns the bytes the call sends to the device."""
    n = len(reqs)
    ra = (_lib.Request * n)(*reqs)
    oa = (_lib.Outputs * n)(*outs)
    h2d = C.c_int64(0)
    call("qcf_batch_prefill", C.byref(model.struct), ra, oa, n, _ptr(ws), ws.numel(),
         C.c_void_p(compute_stream.cuda_stream), C.c_void_p(copy_stream.cuda_stream), C.byref(h2d))
    return int(h2d.value)


def qcf_batch_workspace_size(model, reqs) -> int:
    n = len(reqs)
    ra = (_lib.Request * n)(*reqs)
    return int(_lib.lib().qcf_batch_workspace_size(C.byref(model.struct.dims), ra, n))
