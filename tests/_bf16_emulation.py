"""The oracle's arithmetic with bf16 storage of every GEMM operand (test infrastructure).

The CUDA path keeps the residual stream in fp32 and stores, as bf16 (round to
nearest even), exactly these values: the RMSNorm outputs h and h2, the
projected q, k, v (after RoPE), the attention output o, the SwiGLU activation,
re-rotated chunk keys in the fused cache and the probe's anchor keys.  This
module repeats the oracle's steps with those roundings and nothing else, using
the oracle's own functions for every step.  Its departure from the oracle is
the error that bf16 storage alone forces on any implementation; the parity
tests use it to calibrate the bound where error accumulated through many
layers exceeds the fixed allclose bound (the CUDA path shares no code with it).
"""
from __future__ import annotations

from typing import Dict, List

import numpy as np

from oracle import qcf_oracle as O

F32, F64 = np.float32, np.float64


def bf16(a):
    return O.round_bf16(np.asarray(a, dtype=F32))


def layer(x, W, spec, rope_pos, cache_row, Kc, Vc, capture=None):
    """O.layer_forward with bf16 operands; Kc / Vc updated in place."""
    n = x.shape[0]
    Hq, Hkv, D = spec.n_heads, spec.n_kv_heads, spec.head_dim
    h = bf16(O.rmsnorm(x, W["g_attn"], spec.eps))
    q = bf16(O.rope_rotate((h @ W["wq"].T).reshape(n, Hq, D), rope_pos, spec.theta))
    k = bf16(O.rope_rotate((h @ W["wk"].T).reshape(n, Hkv, D), rope_pos, spec.theta))
    v = bf16((h @ W["wv"].T).reshape(n, Hkv, D))
    if capture is not None:
        capture["q"] = q
    Kc[cache_row] = k
    Vc[cache_row] = v
    o = bf16(O.causal_attention(q, cache_row, Kc, Vc, 1.0 / np.sqrt(D)))
    x = x + o.reshape(n, Hq * D) @ W["wo"].T
    h2 = bf16(O.rmsnorm(x, W["g_mlp"], spec.eps))
    a = bf16(O.silu(h2 @ W["wg"].T) * (h2 @ W["wu"].T))
    return (x + a @ W["wd"].T).astype(F32)


def kv_projection(x, W, spec, positions):
    """O.kv_projection with bf16 storage: fresh post-RoPE K and V of rows x."""
    n = x.shape[0]
    h = bf16(O.rmsnorm(x, W["g_attn"], spec.eps))
    k = bf16(O.rope_rotate((h @ W["wk"].T).reshape(n, spec.n_kv_heads, spec.head_dim), positions, spec.theta))
    v = bf16((h @ W["wv"].T).reshape(n, spec.n_kv_heads, spec.head_dim))
    return k, v


def fused_prefill(model: O.OracleModel, chunk_kv: List[Dict[str, np.ndarray]], context_ids, chunk_start, query_ids,
                  crit: int, n_anchor: int, forced_sel, keep_layers=()) -> Dict[str, object]:
    """O.fused_prefill (critical-layer selector, the given selection) with bf16 storage.

    Re-rotated keys (probe anchors and the fused cache) are stored as bf16, as the
    kernels store them; the LM head reads the last row in fp32, as the kernel does."""
    s = model.spec
    C = int(chunk_start[-1])
    Q = len(query_ids)
    T = C + Q
    n_chunks = len(chunk_kv)
    row_delta = np.repeat(np.asarray(chunk_start[:-1], dtype=np.int64), np.diff(chunk_start))
    K_crit = np.concatenate([ck["K"][crit] for ck in chunk_kv], axis=0)
    anchors = O.keynorm_anchors(K_crit, chunk_start, n_anchor)
    a_rows = np.concatenate([chunk_start[c] + anchors[c] for c in range(n_chunks)]).astype(np.int64)
    a_delta = row_delta[a_rows]
    nA = len(a_rows)
    qpos = C + np.arange(Q)
    x = model.embed_rows(query_ids)
    for l in range(crit):
        Kc = np.zeros((nA + Q, s.n_kv_heads, s.head_dim), dtype=F32)
        Vc = np.zeros_like(Kc)
        aK = np.concatenate([chunk_kv[c]["K"][l][anchors[c]] for c in range(n_chunks)])
        Kc[:nA] = bf16(O.rope_reposition(aK, a_delta, s.theta))
        Vc[:nA] = np.concatenate([chunk_kv[c]["V"][l][anchors[c]] for c in range(n_chunks)])
        x = layer(x, model.layer(l), s, qpos, nA + np.arange(Q), Kc, Vc)
    W = model.layer(crit)
    h = bf16(O.rmsnorm(x, W["g_attn"], s.eps))
    q_crit = bf16(O.rope_rotate((h @ W["wq"].T).reshape(Q, s.n_heads, s.head_dim), qpos, s.theta))

    def K_hat(l):
        return bf16(O.rope_reposition(np.concatenate([ck["K"][l] for ck in chunk_kv]), row_delta, s.theta))

    scores = O.profile_scores(q_crit, K_hat(crit), 1.0 / np.sqrt(s.head_dim))
    sel = np.sort(np.asarray(forced_sel, dtype=np.int64))
    S = np.concatenate([sel, np.arange(C, T)]).astype(np.int64)
    ids_all = np.concatenate([np.asarray(context_ids), np.asarray(query_ids)]).astype(np.int64)
    x = model.embed_rows(ids_all[S])
    K_f, V_f = {}, {}
    for l in range(s.n_layers):
        Kc = np.zeros((T, s.n_kv_heads, s.head_dim), dtype=F32)
        Vc = np.zeros_like(Kc)
        Kc[:C] = K_hat(l)
        Vc[:C] = np.concatenate([ck["V"][l] for ck in chunk_kv])
        x = layer(x, model.layer(l), s, S, S, Kc, Vc)
        if l in keep_layers:
            K_f[l], V_f[l] = Kc, Vc
    return {"q_crit": q_crit, "scores": scores, "x": x, "K": K_f, "V": V_f, **O.lm_head_last(model, x[-1])}


def full_prefill(model: O.OracleModel, ids) -> Dict[str, object]:
    """O.full_prefill with bf16 storage."""
    s = model.spec
    ids = np.asarray(ids, dtype=np.int64)
    T = len(ids)
    rows = np.arange(T)
    x = model.embed_rows(ids)
    Ks, Vs = [], []
    for l in range(s.n_layers):
        Kc = np.zeros((T, s.n_kv_heads, s.head_dim), dtype=F32)
        Vc = np.zeros_like(Kc)
        x = layer(x, model.layer(l), s, rows, rows, Kc, Vc)
        Ks.append(Kc)
        Vs.append(Vc)
    return {"x": x, "K": np.stack(Ks), "V": np.stack(Vs), **O.lm_head_last(model, x[-1])}


def error_stats(got, ref):
    """(max-abs, RMS) of got - ref."""
    d = np.asarray(got, F64) - np.asarray(ref, F64)
    return float(np.max(np.abs(d))) if d.size else 0.0, float(np.sqrt(np.mean(d * d))) if d.size else 0.0
