"""Device model, offline chunk store and per-request driver wrappers.

Weights are packed once into the layout the tensor-core GEMMs read (see
qcf_layer_weights in include/qcf.h); the chunk store keeps every chunk's
per-layer K/V and its anchors in pinned host memory, built with the library's
own full prefill, anchor and gather kernels.
"""
from __future__ import annotations

import ctypes as C
import hashlib
import os
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import _lib
from . import qcf as Q


def _pad_rows(w: torch.Tensor, rows: int) -> torch.Tensor:
    if w.shape[0] == rows:
        return w
    out = torch.zeros((rows,) + tuple(w.shape[1:]), dtype=w.dtype, device=w.device)
    out[: w.shape[0]] = w
    return out


class DeviceModel:
    """A decoder's weights on one GPU, packed for the library, plus its RoPE table.

    `weights` provides .spec, .layer(l) (wq, wk, wv, wo, wg, wu, wd in nn.Linear
    layout, g_attn, g_mlp), .embed(), .lm_head(), .final_norm().
    """

    def __init__(self, weights, device="cuda", max_pos: int = 8192):
        s = weights.spec
        self.spec = s
        self.device = torch.device(device)
        F = s.ffn
        self.ffn_padded = (F + 63) // 64 * 64
        Fp, d = self.ffn_padded, s.d_model
        self.layer_tensors: List[Dict[str, torch.Tensor]] = []
        for l in range(s.n_layers):
            w = {k: v.to(self.device, dtype=torch.bfloat16) for k, v in weights.layer(l).items()}
            gate = _pad_rows(w["wg"], Fp).view(Fp // 64, 64, d)
            up = _pad_rows(w["wu"], Fp).view(Fp // 64, 64, d)
            down = torch.zeros((d, Fp), dtype=torch.bfloat16, device=self.device)
            down[:, :F] = w["wd"]
            packed = {
                "w_qkv": torch.cat([w["wq"], w["wk"], w["wv"]], 0).contiguous(),
                "w_o": w["wo"].contiguous(),
                "w_gu": torch.stack([gate, up], 1).reshape(2 * Fp, d).contiguous(),
                "w_down": down,
                "g_attn": w["g_attn"].contiguous(),
                "g_mlp": w["g_mlp"].contiguous(),
            }
            del w, gate, up
            self.layer_tensors.append(packed)
        self.embed = weights.embed().to(self.device, dtype=torch.bfloat16).contiguous()
        self.lm_head = weights.lm_head().to(self.device, dtype=torch.bfloat16).contiguous()
        self.g_final = weights.final_norm().to(self.device, dtype=torch.bfloat16).contiguous()
        self.rope = Q.RopeTable(max_pos, s.head_dim, s.theta, self.device)
        arr = (_lib.LayerWeights * s.n_layers)()
        for l, t in enumerate(self.layer_tensors):
            arr[l] = _lib.LayerWeights(t["w_qkv"].data_ptr(), t["w_o"].data_ptr(), t["w_gu"].data_ptr(),
                                       t["w_down"].data_ptr(), t["g_attn"].data_ptr(), t["g_mlp"].data_ptr())
        self._layer_arr = arr
        dims = _lib.Dims(s.n_layers, s.d_model, s.n_heads, s.n_kv_heads, s.head_dim, F, Fp, s.vocab, s.eps, s.theta)
        self.struct = _lib.Model(dims, self.embed.data_ptr(), self.lm_head.data_ptr(), self.g_final.data_ptr(),
                                 C.cast(arr, C.POINTER(_lib.LayerWeights)), self.rope.struct)


class StoredChunk:
    def __init__(self, tokens, K, V, anchor_idx, aK, aV):
        self.tokens = tokens          # np.int32 [len]
        self.K, self.V = K, V         # pinned bf16 [L][len][Hkv][D]
        self.anchor_idx = anchor_idx  # np.int32 [A]
        self.aK, self.aV = aK, aV     # pinned bf16 [L][A][Hkv][D]


class ChunkStore:
    """Offline chunk KV (computed alone at positions 0..len-1) and key-norm anchors.

    Chunks are keyed by content: a chunk's stored K/V depends only on its tokens, so a
    chunk id whose tokens were seen before maps to the stored chunk with those tokens
    (the same host arrays, which the batched prefill then copies once per layer).
    """

    def __init__(self, model: DeviceModel, crit_layer: int, n_anchor: int):
        self.model, self.crit, self.n_anchor = model, int(crit_layer), int(n_anchor)
        self.chunks: Dict[int, StoredChunk] = {}
        self.by_content: Dict[bytes, StoredChunk] = {}

    @staticmethod
    def content_key(tokens) -> bytes:
        return hashlib.sha256(np.ascontiguousarray(np.asarray(tokens, dtype=np.int32)).tobytes()).digest()

    def _known(self, chunk_id: int, tokens) -> Optional[StoredChunk]:
        c = self.by_content.get(self.content_key(tokens))
        if c is not None:
            self.chunks[int(chunk_id)] = c
        return c

    def _keep(self, chunk_id: int, c: StoredChunk) -> StoredChunk:
        self.chunks[int(chunk_id)] = c
        self.by_content[self.content_key(c.tokens)] = c
        return c

    def _anchors(self, K_dev: List[torch.Tensor], V_dev: List[torch.Tensor]):
        L = len(K_dev)
        n = K_dev[0].shape[0]
        A = self.n_anchor
        if A == 0:
            z = torch.empty((L, 0) + tuple(K_dev[0].shape[1:]), dtype=torch.bfloat16).pin_memory()
            return np.zeros(0, np.int32), z, z.clone().pin_memory()
        idx = Q.qcf_anchor_keynorm_topk(K_dev[self.crit], [0, n], A)[0].contiguous()
        aK = torch.stack([Q.qcf_gather_rows(K_dev[l], idx) for l in range(L)])
        aV = torch.stack([Q.qcf_gather_rows(V_dev[l], idx) for l in range(L)])
        return idx.cpu().numpy(), aK.cpu().pin_memory(), aV.cpu().pin_memory()

    def ingest(self, chunk_id: int, tokens: np.ndarray) -> StoredChunk:
        """Prefill the chunk alone on the GPU, keep its K/V and anchors in pinned host memory."""
        known = self._known(chunk_id, tokens)
        if known is not None:
            return known
        ids = torch.as_tensor(np.asarray(tokens, dtype=np.int32), device=self.model.device)
        K, V, _, _ = Q.qcf_full_prefill(self.model, ids)
        idx, aK, aV = self._anchors(K, V)
        Kh = torch.stack(K).cpu().pin_memory()
        Vh = torch.stack(V).cpu().pin_memory()
        return self._keep(chunk_id, StoredChunk(np.asarray(tokens, np.int32), Kh, Vh, idx, aK, aV))

    def add_precomputed(self, chunk_id: int, tokens: np.ndarray, K: torch.Tensor, V: torch.Tensor) -> StoredChunk:
        """Store given K/V [L][len][Hkv][D] (bf16, any device) and compute its anchors on the GPU."""
        known = self._known(chunk_id, tokens)
        if known is not None:
            return known
        Kd = [k.to(self.model.device).contiguous() for k in K]
        Vd = [v.to(self.model.device).contiguous() for v in V]
        idx, aK, aV = self._anchors(Kd, Vd)
        return self._keep(chunk_id, StoredChunk(np.asarray(tokens, np.int32),
                                                K.to(torch.bfloat16).cpu().contiguous().pin_memory(),
                                                V.to(torch.bfloat16).cpu().contiguous().pin_memory(), idx, aK, aV))


class ChunkFiles:
    """A storage tier for a chunk store: every stored chunk's per-layer K and V in a file
    (QCFuse 2.A keeps chunk KV on SSD and the anchors in CPU memory).

    File layout, raw bf16: the keys [L][len][Hkv][D], then the values [L][len][Hkv][D].
    Files are named by the chunk's content hash, so a chunk shared by requests is stored
    once.  With o_direct the reads bypass the page cache (where the file system supports
    it and every block is 4096-byte aligned); otherwise they are plain buffered reads.
    """

    ALIGN = 4096

    def __init__(self, store: "ChunkStore", directory: str, o_direct: bool = True):
        self.store, self.directory = store, directory
        os.makedirs(directory, exist_ok=True)
        self.paths: Dict[bytes, str] = {}
        self.fds: Dict[bytes, int] = {}
        self.o_direct_requested = o_direct
        self.o_direct = False

    def write(self, chunk_ids: Sequence[int]) -> int:
        """Writes the chunks not yet on storage; returns the bytes written."""
        written = 0
        for cid in chunk_ids:
            c = self.store.chunks[int(cid)]
            key = ChunkStore.content_key(c.tokens)
            if key in self.paths:
                continue
            path = os.path.join(self.directory, key.hex()[:32] + ".kv")
            with open(path, "wb") as f:
                for t in (c.K, c.V):
                    b = t.contiguous().view(torch.int16).numpy().tobytes()
                    f.write(b)
                    written += len(b)
            self.paths[key] = path
        return written

    def _fd(self, key: bytes) -> int:
        if key not in self.fds:
            flags = os.O_RDONLY
            fd = -1
            if self.o_direct_requested and hasattr(os, "O_DIRECT"):
                try:
                    fd = os.open(self.paths[key], flags | os.O_DIRECT)
                    self.o_direct = True
                except OSError:
                    fd = -1
            if fd < 0:
                fd = os.open(self.paths[key], flags)
                self.o_direct = False
            self.fds[key] = fd
        return self.fds[key]

    def files_for(self, request: "FusedRequest"):
        """qcf_chunk_file entries for the request's chunks, in its retrieval order."""
        s = request.model.spec
        row = s.n_kv_heads * s.head_dim * 2
        arr = (_lib.ChunkFile * len(request.chunks))()
        for i, c in enumerate(request.chunks):
            key = ChunkStore.content_key(c.tokens)
            block = len(c.tokens) * row
            arr[i] = _lib.ChunkFile(self._fd(key), 0, s.n_layers * block, block)
        return arr

    def aligned_for_direct(self, request: "FusedRequest") -> bool:
        s = request.model.spec
        row = s.n_kv_heads * s.head_dim * 2
        starts = np.cumsum([0] + [len(c.tokens) for c in request.chunks])
        sizes = [len(c.tokens) * row for c in request.chunks]
        return all(v % self.ALIGN == 0 for v in sizes + [int(x) * row for x in starts])

    def close(self):
        for fd in self.fds.values():
            os.close(fd)
        self.fds.clear()


SELECT_CRITICAL, SELECT_ALL_LAYERS, SELECT_HKVD = 0, 1, 2


class FusedRequest:
    """Inputs, outputs and workspace of one fused prefill (structs for qcf_request_prefill).

    selector: SELECT_CRITICAL (QCFuse; the store's critical layer, L-1 for QCLast),
    SELECT_ALL_LAYERS (QCAll) or SELECT_HKVD (CacheBlend's KV-deviation selection with
    gradual filtering, kept shares `layer_ratio_bp` [L], non-increasing, ending at ratio_bp).
    """

    def __init__(self, model: DeviceModel, store: ChunkStore, chunk_ids: Sequence[int], query_ids: np.ndarray,
                 ratio_bp: int, forced_sel: Optional[np.ndarray] = None, selector: int = SELECT_CRITICAL,
                 layer_ratio_bp: Optional[Sequence[int]] = None):
        s = model.spec
        dev = model.device
        self.model, self.store = model, store
        chunks = [store.chunks[int(c)] for c in chunk_ids]
        self.chunks = chunks
        self.chunk_ids = [int(c) for c in chunk_ids]
        lens = [len(c.tokens) for c in chunks]
        self.C = int(sum(lens))
        self.Q = len(query_ids)
        self.T = self.C + self.Q
        self.N = Q.qcf_num_selected(self.C, ratio_bp)
        self.ns = self.N + self.Q
        ids = np.concatenate([c.tokens for c in chunks] + [np.asarray(query_ids, np.int32)]).astype(np.int32)
        self.ids_host = torch.from_numpy(ids).pin_memory()
        self.ids = self.ids_host.to(dev)
        self._lens = (C.c_int32 * len(lens))(*lens)
        self._kh = (C.c_void_p * len(chunks))(*[c.K.data_ptr() for c in chunks])
        self._vh = (C.c_void_p * len(chunks))(*[c.V.data_ptr() for c in chunks])
        A = store.n_anchor
        aidx = np.concatenate([c.anchor_idx for c in chunks]).astype(np.int32) if A > 0 else np.zeros(1, np.int32)
        self._aidx = (C.c_int32 * max(1, len(aidx)))(*aidx.tolist())
        self._akh = (C.c_void_p * len(chunks))(*[c.aK.data_ptr() for c in chunks])
        self._avh = (C.c_void_p * len(chunks))(*[c.aV.data_ptr() for c in chunks])
        self.forced = None
        if forced_sel is not None:
            self.forced = torch.as_tensor(np.sort(np.asarray(forced_sel, np.int32)), device=dev)
        self.selector = int(selector)
        self._sched = None
        self.layer_N = None
        if self.selector == SELECT_HKVD:
            if layer_ratio_bp is None or len(layer_ratio_bp) != s.n_layers:
                raise ValueError("HKVD needs one kept share per layer")
            self._sched = (C.c_int32 * s.n_layers)(*[int(v) for v in layer_ratio_bp])
            self.layer_N = [Q.qcf_num_selected(self.C, int(v)) for v in layer_ratio_bp]
        self.req = _lib.Request(len(chunks), self._lens, self._kh, self._vh, A, self._aidx, self._akh, self._avh,
                                self.ids.data_ptr(), self.Q, store.crit, int(ratio_bp),
                                self.forced.data_ptr() if self.forced is not None else None, self.selector,
                                self._sched)
        kv = (self.T, s.n_kv_heads, s.head_dim)
        self.K = [torch.empty(kv, dtype=torch.bfloat16, device=dev) for _ in range(s.n_layers)]
        self.V = [torch.empty(kv, dtype=torch.bfloat16, device=dev) for _ in range(s.n_layers)]
        self.sel = torch.empty(max(1, self.N), dtype=torch.int32, device=dev)
        self.scores = torch.empty(self.C, dtype=torch.float32, device=dev)
        self.q_crit = torch.empty((self.Q, s.n_heads, s.head_dim), dtype=torch.bfloat16, device=dev)
        self.logits = torch.empty(s.vocab, dtype=torch.float32, device=dev)
        self.token = torch.empty(1, dtype=torch.int32, device=dev)
        self.token_host = torch.zeros(1, dtype=torch.int32).pin_memory()
        self.x_rows = torch.empty((self.ns, s.d_model), dtype=torch.float32, device=dev)
        self._kp = (C.c_void_p * s.n_layers)(*[k.data_ptr() for k in self.K])
        self._vp = (C.c_void_p * s.n_layers)(*[v.data_ptr() for v in self.V])
        self.layer_sel = None
        if self.selector == SELECT_HKVD:
            self.layer_sel = torch.zeros((s.n_layers, max(1, self.layer_N[0])), dtype=torch.int32, device=dev)
        self.outs = _lib.Outputs(self._kp, self._vp, self.sel.data_ptr(), self.scores.data_ptr(),
                                 self.q_crit.data_ptr(), self.logits.data_ptr(), self.token.data_ptr(),
                                 self.token_host.data_ptr(), self.x_rows.data_ptr(),
                                 self.layer_sel.data_ptr() if self.layer_sel is not None else None)
        nb = _lib.lib().qcf_request_workspace_size_for(C.byref(model.struct.dims), C.byref(self.req))
        if nb == 0:
            raise ValueError("malformed request (workspace size 0)")
        self.ws = torch.empty(max(256, nb), dtype=torch.uint8, device=dev)

    def run(self, compute_stream=None, copy_stream=None, ids_from_host: bool = False) -> None:
        """Enqueue the fused prefill; with ids_from_host the token ids are copied H2D first."""
        cs = compute_stream or torch.cuda.current_stream()
        xs = copy_stream or cs
        if ids_from_host:
            with torch.cuda.stream(cs):
                self.ids.copy_(self.ids_host, non_blocking=True)
        Q.qcf_request_prefill(self.model, self.req, self.outs, self.ws, cs, xs)

    def run_from_storage(self, files: "ChunkFiles", compute_stream=None, copy_stream=None) -> None:
        """Enqueue the fused prefill with the chunks' K/V read layer by layer from `files`
        (a storage tier) through a pinned double buffer; anchors stay in host memory."""
        cs = compute_stream or torch.cuda.current_stream()
        xs = copy_stream or cs
        nb = _lib.lib().qcf_storage_staging_bytes(C.byref(self.model.struct.dims), C.byref(self.req))
        if nb == 0:
            raise ValueError("malformed request (staging size 0)")
        if getattr(self, "_staging", None) is None or self._staging.numel() < nb + ChunkFiles.ALIGN:
            self._staging = torch.empty(nb + ChunkFiles.ALIGN, dtype=torch.uint8).pin_memory()
        base = self._staging.data_ptr()
        aligned = (base + ChunkFiles.ALIGN - 1) // ChunkFiles.ALIGN * ChunkFiles.ALIGN
        if files.o_direct_requested and not files.aligned_for_direct(self):
            raise ValueError("O_DIRECT reads need 4096-byte aligned chunk blocks; open ChunkFiles with o_direct=False")
        self._files = files.files_for(self)
        Q.call("qcf_request_prefill_storage", C.byref(self.model.struct), C.byref(self.req), self._files,
               C.c_void_p(aligned), nb, C.byref(self.outs), Q._ptr(self.ws), self.ws.numel(), Q._stream(cs),
               Q._stream(xs))

    @property
    def selected(self) -> torch.Tensor:
        return self.sel[: self.N]


def run_batch(requests: Sequence["FusedRequest"], compute_stream=None, copy_stream=None) -> int:
    """Enqueue several fused prefills whose shared chunks cross the host link once per
    layer; every request's outputs land in its own FusedRequest.  Returns the bytes sent."""
    reqs = list(requests)
    model = reqs[0].model
    cs = compute_stream or torch.cuda.current_stream()
    xs = copy_stream or cs
    structs = [r.req for r in reqs]
    nb = Q.qcf_batch_workspace_size(model, structs)
    if nb == 0:
        raise ValueError("malformed batch (workspace size 0)")
    ws = Q.workspace(nb, model.device, tag="batch")
    return Q.qcf_batch_prefill(model, structs, [r.outs for r in reqs], ws, cs, xs)
