"""CPU oracle for query-centric KV-cache fusion (QCFuse) prefill.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline / reference leg may import or run this module.  The product path
(the CUDA library and its Python binding) never imports it, and it imports
nothing of the product path: the two share only the seeded inputs of `qcfdata`.

What it computes, step by step in the pages' order:

* the Llama-style decoder that both the full-recompute baseline and the fused
  path run (RMSNorm, RoPE, causal GQA attention, SwiGLU), "Full KV Recompute"
  in *CacheBlend problem definition* (section 2.2);
* offline chunk KV precompute at local positions 0..L-1 and semantic-summary
  anchors by key norm (*QCFuse*, technical summary, section 2.A "Anchor-based
  Lightweight Query Probing");
* positional re-rotation of reused chunk keys ("adjust positional encoding",
  *CacheBlend problem definition*, section 2.4 "Full KV Reuse");
* the anchor-prefixed query probe and critical-layer attention profiling with
  top-N selection (*QCFuse*, section 2.A "Critical-layer Attention Profiling");
* per-layer selective recompute of the selected rows with location-aware
  causal attention over the fused cache (*QCFuse*, section 2.A "pipelined cache
  reconstruction" and its sparse attention kernel; *KVCache reuse 01*, section
  1.3.4 "selective recompute flow");
* the selector variants the pages compare against: QCLast (profiling at the
  last layer) and QCAll (query-aware profiling at every layer), *QCFuse*,
  section 4 "Results"; CacheBlend's KV-deviation selection with gradual
  filtering across layers (*KVCache reuse 01*, sections 1.3.2-1.3.4).

Precision: matmuls in fp32; RoPE angles, softmax normalisers, score sums,
RMSNorm statistics and the final logits in fp64.  Stored chunk K/V can be
rounded to bf16 (round to nearest even) to model the cache's storage format.

Readings where the pages are silent (the plainest one the rest supports):
anchors by the critical layer's key L2 norm over all KV heads; anchors enter the
probe as a KV prefix at their absolute fused positions; the probe runs layers
0..crit-1 and then crit's RMSNorm, W_q and RoPE; profiling softmax runs over the
C context keys only and sums over all query rows and heads; N = ceil(ratio*C)
from basis points; ties go to the lower index; one selection is reused at every
layer; query rows are always recomputed; RoPE is rotate-half with
omega_k = theta^(-2k/D); re-rotation applies R(offset) to the stored key;
fresh K/V of the recomputed rows are written into the cache before attention.
QCLast is the critical-layer selector with crit = L-1; QCAll keeps the anchors,
runs the probe through layers 0..L-2 and sums the per-layer profile scores of
all L layers (each layer's q from the probe against that layer's re-rotated
keys), then selects once.  HKVD: a token's KV deviation at a layer is the
squared L2 distance between its fresh and its reused K and V over all KV heads
(the ranking of the L2 distance); at layer 0 every context token is measured,
at layer l the tokens kept after layer l-1; the kept set at layer l is the
top ceil(r_l*C) of those by deviation (ties to the lower position), and only
the kept rows and the query get fresh K/V, attention and MLP at that layer.

Parity unpinned against the pages for those readings: no printed value decides
them.  The tests pin the arithmetic to closed forms, library routines and the
special cases the pages state (full recompute, prefix caching, full reuse).
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

F32 = np.float32
F64 = np.float64


# --------------------------------------------------------------------------- helpers

def as_f32(a) -> np.ndarray:
    """Convert a numpy array or a CPU torch tensor (any float dtype) to fp32 numpy."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu")
        if str(a.dtype) != "torch.float32":
            a = a.float()
        a = a.numpy()
    return np.ascontiguousarray(a, dtype=F32)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bfloat16 (ties to even), kept as fp32.

    bfloat16 keeps the top 16 bits of the fp32 pattern; adding 0x7FFF plus the
    lowest kept bit before truncation rounds to nearest with ties to even.
    """
    u = np.ascontiguousarray(a, dtype=F32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(F32)


class OracleModel:
    """fp32 view of a weight source with `.spec`, `.layer(l)`, `.embed()`,
    `.lm_head()` and `.final_norm()` (tensors in nn.Linear [out][in] layout).

    Small models are cached whole; large ones are converted layer by layer.
    """

    def __init__(self, weights, cache: Optional[bool] = None):
        self.src = weights
        self.spec = weights.spec
        s = self.spec
        params = s.n_layers * (s.d_model * (2 * s.q_width + 2 * s.kv_width) + 3 * s.d_model * s.ffn)
        self.cache = params < 50_000_000 if cache is None else cache
        self._layers: Dict[int, Dict[str, np.ndarray]] = {}
        self._embed = None
        self._lm = None

    def layer(self, l: int) -> Dict[str, np.ndarray]:
        if l in self._layers:
            return self._layers[l]
        w = {k: as_f32(v) for k, v in self.src.layer(l).items()}
        if self.cache:
            self._layers[l] = w
        return w

    def embed_rows(self, ids: np.ndarray) -> np.ndarray:
        if self._embed is None:
            self._embed = as_f32(self.src.embed())
        return self._embed[np.asarray(ids, dtype=np.int64)].copy()

    def lm_head(self) -> np.ndarray:
        if self._lm is None:
            self._lm = as_f32(self.src.lm_head())
        return self._lm

    def final_norm(self) -> np.ndarray:
        return as_f32(self.src.final_norm())


# --------------------------------------------------------------------------- decoder pieces

def rope_angles(positions: np.ndarray, D: int, theta: float) -> np.ndarray:
    """Angles pos * omega_k, omega_k = theta^(-2k/D), k < D/2, in fp64: [n][D/2]."""
    k = np.arange(D // 2, dtype=F64)
    omega = 1.0 / np.power(F64(theta), 2.0 * k / D)
    return np.asarray(positions, dtype=F64)[:, None] * omega[None, :]


def rope_rotate(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE: pair (k, k+D/2) of every head turns by pos*omega_k.

    x: [n][H][D]; positions: [n] (any integer, including a re-rotation delta).
    """
    D = x.shape[-1]
    ang = rope_angles(positions, D, theta)
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    xd = x.astype(F64)
    a, b = xd[..., : D // 2], xd[..., D // 2:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1).astype(F32)


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g per row, statistics in fp64."""
    xd = x.astype(F64)
    ms = np.mean(xd * xd, axis=-1, keepdims=True)
    return (xd / np.sqrt(ms + eps) * g.astype(F64)).astype(F32)


def silu(z: np.ndarray) -> np.ndarray:
    zd = z.astype(F64)
    return (zd / (1.0 + np.exp(-zd))).astype(F32)


def causal_attention(q: np.ndarray, bound: np.ndarray, K: np.ndarray, V: np.ndarray,
                     scale: float, block: int = 64) -> np.ndarray:
    """Location-aware causal GQA attention over a key/value cache.

    Row r (query head h) attends to every cache row j <= bound[r] with
    softmax_j(scale * q[r,h] . K[j, h // G]) and returns the weighted sum of V.
    This is the computation of the sparse attention kernel of the QCFuse
    summary (section 2.A: a discrete index table, causality by true position)
    and, with bound = arange(T), plain dense causal attention.
    q: [n][Hq][D]; bound: [n]; K, V: [T][Hkv][D].  Arithmetic in fp64.
    """
    n, Hq, D = q.shape
    T, Hkv, _ = K.shape
    G = Hq // Hkv
    keys = np.arange(T)
    out = np.empty((n, Hq, D), dtype=F32)
    for g in range(Hkv):                      # one KV head at a time keeps memory at O(T*D)
        Kg = K[:, g, :].astype(F64)           # [T][D]
        Vg = V[:, g, :].astype(F64)
        for h in range(g * G, (g + 1) * G):
            for r0 in range(0, n, block):
                r1 = min(n, r0 + block)
                s = (q[r0:r1, h, :].astype(F64) @ Kg.T) * scale          # [b][T]
                hidden = keys[None, :] > np.asarray(bound[r0:r1])[:, None]
                s = np.where(hidden, -np.inf, s)
                m = s.max(axis=-1, keepdims=True)
                p = np.exp(s - m)
                p /= p.sum(axis=-1, keepdims=True)
                out[r0:r1, h, :] = (p @ Vg).astype(F32)
    return out


def layer_forward(x: np.ndarray, W: Dict[str, np.ndarray], spec, rope_pos: np.ndarray,
                  cache_row: np.ndarray, Kc: np.ndarray, Vc: np.ndarray,
                  capture: Optional[dict] = None) -> np.ndarray:
    """One decoder layer for the rows of `x` (recomputed rows only).

    Steps, as in the selective recompute flow (*KVCache reuse 01*, 1.3.4):
    RMSNorm -> Q,K,V projections -> RoPE at each row's absolute position ->
    write the fresh K,V into the cache at `cache_row` (before attention) ->
    attention of each row over cache rows <= its own cache row -> O projection
    and residual -> RMSNorm -> SwiGLU MLP and residual.  Kc / Vc are updated in
    place; the new x is returned.  `capture`, when given, receives the
    post-RoPE q.
    """
    n = x.shape[0]
    Hq, Hkv, D = spec.n_heads, spec.n_kv_heads, spec.head_dim
    h = rmsnorm(x, W["g_attn"], spec.eps)
    q = (h @ W["wq"].T).reshape(n, Hq, D)
    k = (h @ W["wk"].T).reshape(n, Hkv, D)
    v = (h @ W["wv"].T).reshape(n, Hkv, D)
    q = rope_rotate(q, rope_pos, spec.theta)
    k = rope_rotate(k, rope_pos, spec.theta)
    if capture is not None:
        capture["q"] = q
    Kc[cache_row] = k
    Vc[cache_row] = v
    o = causal_attention(q, cache_row, Kc, Vc, 1.0 / np.sqrt(D))
    x = x + o.reshape(n, Hq * D) @ W["wo"].T
    h2 = rmsnorm(x, W["g_mlp"], spec.eps)
    a = silu(h2 @ W["wg"].T) * (h2 @ W["wu"].T)
    return (x + a @ W["wd"].T).astype(F32)


def lm_head_last(model: OracleModel, x_last: np.ndarray) -> Dict[str, object]:
    """Final RMSNorm of the last row, fp64 logits, first token = argmax (lowest index)."""
    h = rmsnorm(x_last[None, :], model.final_norm(), model.spec.eps)[0].astype(F64)
    logits = model.lm_head().astype(F64) @ h
    return {"logits": logits, "token": int(np.argmax(logits))}


# --------------------------------------------------------------------------- full recompute

def full_prefill(model: OracleModel, ids: Sequence[int], positions: Optional[np.ndarray] = None,
                 keep_kv: bool = True, capture_q_layer: Optional[int] = None) -> Dict[str, object]:
    """Plain prefill of all tokens ("Full KV Recompute", CacheBlend problem definition 2.2).

    Returns per-layer post-RoPE K/V [L][T][Hkv][D] (when keep_kv), the final
    hidden states, the last row's logits and the first token.
    """
    s = model.spec
    ids = np.asarray(ids, dtype=np.int64)
    T = len(ids)
    pos = np.arange(T) if positions is None else np.asarray(positions)
    rows = np.arange(T)
    x = model.embed_rows(ids)
    Ks, Vs = [], []
    cap: Dict[str, np.ndarray] = {}
    for l in range(s.n_layers):
        Kc = np.zeros((T, s.n_kv_heads, s.head_dim), dtype=F32)
        Vc = np.zeros_like(Kc)
        x = layer_forward(x, model.layer(l), s, pos, rows, Kc, Vc,
                          capture=cap if l == capture_q_layer else None)
        if keep_kv:
            Ks.append(Kc)
            Vs.append(Vc)
    out = {"x": x, **lm_head_last(model, x[-1])}
    if capture_q_layer is not None:
        out["q"] = cap["q"]
    if keep_kv:
        out["K"] = np.stack(Ks)
        out["V"] = np.stack(Vs)
    return out


def chunk_precompute(model: OracleModel, chunk_ids: Sequence[int], store_bf16: bool = True) -> Dict[str, np.ndarray]:
    """Offline KV of one chunk prefilled alone at local positions 0..L-1.

    (*QCFuse* 2.A: chunks are precomputed independently; *CacheBlend problem
    definition* 2.4.)  Stored K/V are rounded to bf16 when `store_bf16`.
    """
    r = full_prefill(model, chunk_ids)
    K, V = r["K"], r["V"]
    if store_bf16:
        K, V = round_bf16(K), round_bf16(V)
    return {"K": K, "V": V}


# --------------------------------------------------------------------------- fusion steps

def rope_reposition(K_stored: np.ndarray, delta: np.ndarray, theta: float) -> np.ndarray:
    """Move stored keys to new absolute positions: K_new = R(delta) K_stored.

    One rotation by the offset delta (rotations compose additively), for keys
    precomputed at local positions and reused at position offset + i.
    K_stored: [n][Hkv][D]; delta: [n] (or a scalar broadcast to every row).
    """
    delta = np.broadcast_to(np.asarray(delta), (K_stored.shape[0],))
    return rope_rotate(K_stored, delta, theta)


def keynorm_anchors(K_crit: np.ndarray, chunk_start: np.ndarray, n_anchor: int) -> np.ndarray:
    """Semantic-summary anchors: per chunk, the n_anchor tokens of largest key norm.

    (*QCFuse* 2.A "Anchor-based Lightweight Query Probing".)  The norm is the L2
    norm of the token's key over all KV heads and head dims at the critical
    layer, in fp64; ties go to the lower index; indices are chunk-local and
    returned ascending: [n_chunks][n_anchor] (fewer if a chunk is shorter).
    """
    out = []
    for c in range(len(chunk_start) - 1):
        rows = K_crit[chunk_start[c]:chunk_start[c + 1]].astype(F64)
        norm = np.sqrt(np.sum(rows.reshape(rows.shape[0], -1) ** 2, axis=1))
        order = np.argsort(-norm, kind="stable")[:n_anchor]
        out.append(np.sort(order))
    return np.asarray(out, dtype=np.int64)


def profile_scores(q: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """Critical-layer attention profiling (*QCFuse* 2.A).

    For every query row r and head h, p_{r,h,j} = softmax_j(scale * q[r,h] . K[j, h//G])
    over the C context keys; score_j = sum_{r,h} p_{r,h,j}.  fp64 throughout.
    q: [nq][Hq][D]; K: [C][Hkv][D] -> scores [C] (fp64).
    """
    nq, Hq, D = q.shape
    C, Hkv, _ = K.shape
    G = Hq // Hkv
    Kh = K.astype(F64)[:, np.arange(Hq) // G, :].transpose(1, 2, 0)  # [Hq][D][C]
    s = np.matmul(q.astype(F64).transpose(1, 0, 2), Kh) * scale        # [Hq][nq][C]
    s -= s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=-1, keepdims=True)
    return p.sum(axis=(0, 1))


def num_selected(C: int, ratio_bp: int) -> int:
    """N = ceil(ratio * C) with the ratio in basis points, clamped to [0, C]."""
    return max(0, min(C, (int(ratio_bp) * int(C) + 9999) // 10000))


def topn_select(scores: np.ndarray, N: int) -> np.ndarray:
    """Indices of the N largest scores (stable order by -score, so ties keep the
    lower index), returned ascending."""
    order = np.argsort(-np.asarray(scores, dtype=F64), kind="stable")[:N]
    return np.sort(order).astype(np.int64)


def anchor_probe(model: OracleModel, query_ids: np.ndarray, anchor_K: List[np.ndarray],
                 anchor_V: List[np.ndarray], anchor_delta: np.ndarray, context_len: int,
                 crit: int, collect_q: Optional[List[np.ndarray]] = None) -> np.ndarray:
    """Context-aware query representation at the critical layer (*QCFuse* 2.A).

    The query rows (absolute positions C..C+Q-1) run layers 0..crit-1 with a KV
    prefix made of the anchors' stored K/V (K re-rotated by its chunk offset to
    its absolute position); query row i attends to every anchor and to query
    rows <= i.  At layer `crit` only RMSNorm, W_q and RoPE run: returns q_crit
    [Q][Hq][D].  anchor_K/V: per layer l < crit, [nA][Hkv][D].  `collect_q`,
    when given, receives the post-RoPE q of every probe layer l < crit.
    """
    s = model.spec
    Q = len(query_ids)
    nA = len(anchor_delta)
    qpos = context_len + np.arange(Q)
    rows = nA + np.arange(Q)
    x = model.embed_rows(query_ids)
    for l in range(crit):
        Kc = np.zeros((nA + Q, s.n_kv_heads, s.head_dim), dtype=F32)
        Vc = np.zeros_like(Kc)
        if nA:
            Kc[:nA] = rope_reposition(anchor_K[l], anchor_delta, s.theta)
            Vc[:nA] = anchor_V[l]
        cap: Dict[str, np.ndarray] = {}
        x = layer_forward(x, model.layer(l), s, qpos, rows, Kc, Vc, capture=cap)
        if collect_q is not None:
            collect_q.append(cap["q"])
    W = model.layer(crit)
    h = rmsnorm(x, W["g_attn"], s.eps)
    q = (h @ W["wq"].T).reshape(Q, s.n_heads, s.head_dim)
    return rope_rotate(q, qpos, s.theta)


def fused_prefill(model: OracleModel, chunk_kv: List[Dict[str, np.ndarray]], context_ids: np.ndarray,
                  chunk_start: np.ndarray, query_ids: np.ndarray, crit: int, ratio_bp: int,
                  n_anchor: int, forced_sel: Optional[np.ndarray] = None,
                  keep_layers: bool = True, layers: Optional[int] = None,
                  selector: str = "critical") -> Dict[str, object]:
    """The whole fused prefill of one request.

    chunk_kv[c] holds the stored K, V [L][L_c][Hkv][D] of the c-th retrieved
    chunk (retrieval order); context_ids are the chunks' tokens concatenated;
    chunk_start[c] = offset of chunk c (prefix sums of lengths).

    1. anchors: top key-norm tokens of each chunk at the critical layer;
    2. probe: q_crit from the query with the anchors as KV prefix;
    3. profile: scores of the C context tokens from the re-rotated critical-layer K;
    4. select: top N = ceil(ratio*C) (or `forced_sel`), plus all query rows;
    5. for every layer: the fused cache is the re-rotated chunk K and stored V;
       the selected rows and the query are recomputed (layer 0 from the
       embeddings) with their fresh K/V written into the cache first;
    6. logits of the last query row and the first token.
    `layers` truncates step 5 (for timing samples); then no logits are produced.
    selector "critical" profiles at `crit` (QCLast: crit = L-1); "all" (QCAll)
    keeps the anchors chosen at `crit`, runs the probe through layers 0..L-2 and
    sums the profile scores of every layer before selecting.
    """
    s = model.spec
    C = int(chunk_start[-1])
    Q = len(query_ids)
    T = C + Q
    n_chunks = len(chunk_kv)
    off = np.asarray(chunk_start[:-1], dtype=np.int64)
    row_delta = np.repeat(off, np.diff(chunk_start))

    K_crit_stored = np.concatenate([ck["K"][crit] for ck in chunk_kv], axis=0)
    anchors = keynorm_anchors(K_crit_stored, chunk_start, n_anchor)
    a_rows = np.concatenate([chunk_start[c] + anchors[c] for c in range(n_chunks)]).astype(np.int64)
    a_delta = row_delta[a_rows]
    assert selector in ("critical", "all")
    depth = crit if selector == "critical" else s.n_layers - 1   # probe layers before the last profiled one
    aK = [np.concatenate([chunk_kv[c]["K"][l][anchors[c]] for c in range(n_chunks)]) for l in range(depth)]
    aV = [np.concatenate([chunk_kv[c]["V"][l][anchors[c]] for c in range(n_chunks)]) for l in range(depth)]
    q_layers: List[np.ndarray] = []
    q_crit = anchor_probe(model, query_ids, aK, aV, a_delta, C, depth, collect_q=q_layers)
    scale = 1.0 / np.sqrt(s.head_dim)

    def K_hat(l):
        return rope_reposition(np.concatenate([ck["K"][l] for ck in chunk_kv], axis=0), row_delta, s.theta)

    if selector == "critical":
        scores = profile_scores(q_crit, K_hat(crit), scale)
    else:   # QCAll: every layer's query-to-context profile, summed
        scores = profile_scores(q_crit, K_hat(depth), scale)
        for l in range(depth):
            scores = scores + profile_scores(q_layers[l], K_hat(l), scale)
    N = num_selected(C, ratio_bp)
    sel = topn_select(scores, N) if forced_sel is None else np.sort(np.asarray(forced_sel, dtype=np.int64))
    S = np.concatenate([sel, np.arange(C, T)]).astype(np.int64)

    ids_all = np.concatenate([np.asarray(context_ids), np.asarray(query_ids)]).astype(np.int64)
    x = model.embed_rows(ids_all[S])
    K_f, V_f, xs = [], [], []
    n_run = s.n_layers if layers is None else layers
    for l in range(n_run):
        Kc = np.zeros((T, s.n_kv_heads, s.head_dim), dtype=F32)
        Vc = np.zeros_like(Kc)
        Kc[:C] = rope_reposition(np.concatenate([ck["K"][l] for ck in chunk_kv]), row_delta, s.theta)
        Vc[:C] = np.concatenate([ck["V"][l] for ck in chunk_kv])
        x = layer_forward(x, model.layer(l), s, S, S, Kc, Vc)
        if keep_layers:
            K_f.append(Kc)
            V_f.append(Vc)
            xs.append(x.copy())
    out = {"anchors": anchors, "anchor_rows": a_rows, "q_crit": q_crit, "scores": scores,
           "N": N, "sel": sel, "rows": S, "x": x}
    if layers is None:
        out.update(lm_head_last(model, x[-1]))
    if keep_layers:
        out.update({"K": np.stack(K_f), "V": np.stack(V_f), "x_layers": xs})
    return out


# --------------------------------------------------------------------------- CacheBlend HKVD selection

def kv_projection(x: np.ndarray, W: Dict[str, np.ndarray], spec, positions: np.ndarray):
    """Fresh post-RoPE K and V of rows x at `positions` (the K/V part of a layer)."""
    n = x.shape[0]
    h = rmsnorm(x, W["g_attn"], spec.eps)
    k = (h @ W["wk"].T).reshape(n, spec.n_kv_heads, spec.head_dim)
    v = (h @ W["wv"].T).reshape(n, spec.n_kv_heads, spec.head_dim)
    return rope_rotate(k, positions, spec.theta), v


def kv_deviation(k: np.ndarray, v: np.ndarray, K_reused: np.ndarray, V_reused: np.ndarray) -> np.ndarray:
    """Per row: squared L2 distance between fresh and reused K and V over all heads
    (*KVCache reuse 01*, 1.3.2 "KV Deviation"), fp64."""
    dk = np.asarray(k, dtype=F64) - np.asarray(K_reused, dtype=F64)
    dv = np.asarray(v, dtype=F64) - np.asarray(V_reused, dtype=F64)
    return (dk * dk).sum(axis=(1, 2)) + (dv * dv).sum(axis=(1, 2))


def hkvd_prefill(model: OracleModel, chunk_kv: List[Dict[str, np.ndarray]], context_ids: np.ndarray,
                 chunk_start: np.ndarray, query_ids: np.ndarray, layer_ratio_bp: Sequence[int],
                 forced_layer_sel: Optional[List[np.ndarray]] = None,
                 keep_layers: bool = True) -> Dict[str, object]:
    """Fused prefill with CacheBlend's KV-deviation selection and gradual filtering
    (*KVCache reuse 01*, 1.3.3 "three-level token selection" and 1.3.4).

    Layer l measures the KV deviation of the context rows kept after layer l-1
    (every context row at layer 0), keeps the top ceil(r_l*C) of them
    (`layer_ratio_bp[l]`, non-increasing), gives those rows and the query fresh
    K/V in the fused cache, and runs attention and the MLP for them only.
    `forced_layer_sel[l]`, when given, replaces layer l's choice (positions,
    ascending, a subset of the rows kept after layer l-1).
    """
    s = model.spec
    C = int(chunk_start[-1])
    Q = len(query_ids)
    T = C + Q
    row_delta = np.repeat(np.asarray(chunk_start[:-1], dtype=np.int64), np.diff(chunk_start))
    ids_all = np.concatenate([np.asarray(context_ids), np.asarray(query_ids)]).astype(np.int64)
    qrows = np.arange(C, T)
    prev = np.arange(C)
    x = model.embed_rows(ids_all[np.concatenate([prev, qrows])])
    devs, sels, K_f, V_f = [], [], [], []
    for l in range(s.n_layers):
        W = model.layer(l)
        Kc = np.zeros((T, s.n_kv_heads, s.head_dim), dtype=F32)
        Vc = np.zeros_like(Kc)
        Kc[:C] = rope_reposition(np.concatenate([ck["K"][l] for ck in chunk_kv]), row_delta, s.theta)
        Vc[:C] = np.concatenate([ck["V"][l] for ck in chunk_kv])
        pos_prev = np.concatenate([prev, qrows])
        k, v = kv_projection(x, W, s, pos_prev)
        dev = kv_deviation(k[:len(prev)], v[:len(prev)], Kc[prev], Vc[prev])
        N = num_selected(C, int(layer_ratio_bp[l]))
        assert N <= len(prev), "the ratio schedule must not increase"
        if forced_layer_sel is None:
            keep = topn_select(dev, N)
        else:
            keep = np.searchsorted(prev, np.asarray(forced_layer_sel[l], dtype=np.int64))
            assert len(keep) == N and np.array_equal(prev[keep], np.sort(forced_layer_sel[l]))
        keep_idx = np.concatenate([keep, len(prev) + np.arange(Q)])
        rows = pos_prev[keep_idx]
        x = layer_forward(x[keep_idx], W, s, rows, rows, Kc, Vc)
        prev = prev[keep]
        devs.append(dev)
        sels.append(prev.copy())
        if keep_layers:
            K_f.append(Kc)
            V_f.append(Vc)
    out = {"layer_dev": devs, "layer_sel": sels, "sel": prev, "x": x, **lm_head_last(model, x[-1])}
    if keep_layers:
        out.update({"K": np.stack(K_f), "V": np.stack(V_f)})
    return out
