"""Pins of the CPU oracle to things other than itself (CPU only).

Each test ties one oracle function to a closed form, a library routine, a
brute-force loop on tiny inputs, or a special case the pages state:
  * full recompute == the plain decoder (CacheBlend problem definition 2.2);
  * prefix caching reproduces full recompute on the first chunk (2.3);
  * full KV reuse only re-rotates stored keys (2.4);
  * ratio 1 recomputes everything, so fusion == full recompute.
"""
import dataclasses
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import qcfdata as qd
from oracle import qcf_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def tiny():
    return O.OracleModel(qd.ModelWeights(qd.TINY))


def tiny_request(n_chunks=3, chunk_len=32, Q=8, chunk_ids=None):
    s = qd.TINY
    ids = list(range(n_chunks)) if chunk_ids is None else chunk_ids
    chunks = [qd.chunk_tokens(c, chunk_len, s.vocab) for c in ids]
    start = np.arange(len(ids) + 1) * chunk_len
    return chunks, start, qd.query_tokens(0, Q, s.vocab)


# ----------------------------------------------------------------- RoPE

def test_rope_unit_vector_is_rotate_half():
    D = 16
    x = np.zeros((1, 1, D), np.float32)
    x[0, 0, 0] = 1.0
    y = O.rope_rotate(x, np.array([1]), 1e4)[0, 0]
    want = np.zeros(D)
    want[0], want[D // 2] = math.cos(1.0), math.sin(1.0)   # 2-D rotation of (1, 0) by 1 rad
    np.testing.assert_allclose(y, want, atol=1e-7)


def test_rope_frequency_ladder():
    # omega_k = theta^(-2k/D): at k = D/4 and theta = 1e4 the frequency is 1/100.
    D = 16
    k = D // 4
    x = np.zeros((1, 1, D), np.float32)
    x[0, 0, k] = 1.0
    y = O.rope_rotate(x, np.array([100]), 1e4)[0, 0]
    assert abs(y[k] - math.cos(1.0)) < 1e-6 and abs(y[k + D // 2] - math.sin(1.0)) < 1e-6
    assert np.count_nonzero(np.abs(y) > 1e-9) == 2


def test_rope_is_relative_and_orthogonal():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, 2, 128)).astype(np.float32)
    k = rng.standard_normal((1, 2, 128)).astype(np.float32)
    for p, pk, d in [(5, 3, 100), (4000, 17, 70000), (0, 0, 131071)]:
        a = np.sum(O.rope_rotate(q, np.array([p]), 1e4) * O.rope_rotate(k, np.array([pk]), 1e4))
        b = np.sum(O.rope_rotate(q, np.array([p + d]), 1e4) * O.rope_rotate(k, np.array([pk + d]), 1e4))
        assert abs(a - b) < 1e-3 * max(1.0, abs(a))
    r = O.rope_rotate(q, np.array([12345]), 1e4)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(q, axis=-1), rtol=1e-6)


def test_reposition_composes_rotations():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((6, 4, 16)).astype(np.float32)
    local = np.arange(6)
    stored = O.rope_rotate(x, local, 1e4)
    moved = O.rope_reposition(stored, np.full(6, 777), 1e4)
    direct = O.rope_rotate(x, local + 777, 1e4)
    np.testing.assert_allclose(moved, direct, atol=2e-6)
    np.testing.assert_array_equal(O.rope_reposition(stored, 0, 1e4), stored)


# ----------------------------------------------------------------- norms, attention

def test_rmsnorm_closed_form():
    y = O.rmsnorm(np.array([[3.0, 4.0]], np.float32), np.ones(2, np.float32), 1e-5)
    np.testing.assert_allclose(y[0], np.array([3.0, 4.0]) / math.sqrt(12.5 + 1e-5), rtol=1e-7)
    x = np.random.default_rng(2).standard_normal((5, 64)).astype(np.float32) * 7
    y = O.rmsnorm(x, np.ones(64, np.float32), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y.astype(np.float64) ** 2, axis=1)), 1.0, rtol=1e-6)


def _sdpa_reference(q, bound, K, V, scale):
    n, Hq, D = q.shape
    T, Hkv, _ = K.shape
    G = Hq // Hkv
    qt = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]
    kt = torch.from_numpy(K.astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    vt = torch.from_numpy(V.astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    mask = torch.arange(T)[None, :] <= torch.from_numpy(np.asarray(bound))[:, None]
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def test_attention_matches_library_sdpa():
    rng = np.random.default_rng(3)
    T, Hq, Hkv, D = 70, 8, 2, 16
    K = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    V = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    rows = np.sort(rng.choice(T, 23, replace=False))
    q = rng.standard_normal((len(rows), Hq, D)).astype(np.float32)
    got = O.causal_attention(q, rows, K, V, 0.25, block=7)
    np.testing.assert_allclose(got, _sdpa_reference(q, rows, K, V, 0.25), atol=1e-6)


def test_attention_special_cases():
    rng = np.random.default_rng(4)
    K = rng.standard_normal((9, 2, 8)).astype(np.float32)
    V = rng.standard_normal((9, 2, 8)).astype(np.float32)
    q = rng.standard_normal((3, 4, 8)).astype(np.float32)
    o = O.causal_attention(q, np.array([0, 0, 0]), K, V, 1.0)   # one visible key
    np.testing.assert_allclose(o[:, 0], np.broadcast_to(V[0, 0], (3, 8)), atol=1e-6)
    np.testing.assert_allclose(o[:, 3], np.broadcast_to(V[0, 1], (3, 8)), atol=1e-6)
    o = O.causal_attention(q, np.array([8, 8, 8]), K, np.ones_like(V), 1.0)  # rows of p sum to 1
    np.testing.assert_allclose(o, 1.0, atol=1e-6)


# ----------------------------------------------------------------- decoder

def _torch_decoder(model, ids, n_layers):
    """Independent fp64 decoder from library routines: F.rms_norm, F.linear,
    F.scaled_dot_product_attention(is_causal), F.silu, RoPE by complex multiplication."""
    s = model.spec
    T = len(ids)
    x = torch.from_numpy(model.embed_rows(ids).astype(np.float64))
    half = s.head_dim // 2
    inv = 1.0 / (s.theta ** (torch.arange(half, dtype=torch.float64) * 2 / s.head_dim))
    rot = torch.polar(torch.ones(T, half, dtype=torch.float64), torch.arange(T, dtype=torch.float64)[:, None] * inv)

    def rope(t):   # t [T][H][D]; pair (k, k + D/2) as a complex number
        z = torch.complex(t[..., :half], t[..., half:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    G = s.n_heads // s.n_kv_heads
    for l in range(n_layers):
        W = {k: torch.from_numpy(v.astype(np.float64)) for k, v in model.layer(l).items()}
        h = F.rms_norm(x, (s.d_model,), W["g_attn"], s.eps)
        q = rope(F.linear(h, W["wq"]).view(T, s.n_heads, s.head_dim))
        k = rope(F.linear(h, W["wk"]).view(T, s.n_kv_heads, s.head_dim))
        v = F.linear(h, W["wv"]).view(T, s.n_kv_heads, s.head_dim)
        o = F.scaled_dot_product_attention(q.transpose(0, 1)[None], k.transpose(0, 1).repeat_interleave(G, 0)[None],
                                           v.transpose(0, 1).repeat_interleave(G, 0)[None], is_causal=True)
        x = x + F.linear(o[0].transpose(0, 1).reshape(T, -1), W["wo"])
        h2 = F.rms_norm(x, (s.d_model,), W["g_mlp"], s.eps)
        x = x + F.linear(F.silu(F.linear(h2, W["wg"])) * F.linear(h2, W["wu"]), W["wd"])
    hl = F.rms_norm(x[-1], (s.d_model,), torch.from_numpy(model.final_norm().astype(np.float64)), s.eps)
    return x.numpy(), (torch.from_numpy(model.lm_head().astype(np.float64)) @ hl).numpy()


def test_full_prefill_matches_library_decoder(tiny):
    ids = qd.token_ids(40, qd.TINY.vocab, stream=99)
    r = O.full_prefill(tiny, ids)
    x_ref, logits_ref = _torch_decoder(tiny, ids, qd.TINY.n_layers)
    np.testing.assert_allclose(r["x"], x_ref, atol=2e-5, rtol=1e-5)
    np.testing.assert_allclose(r["logits"], logits_ref, atol=2e-5, rtol=1e-5)
    assert r["token"] == int(np.argmax(logits_ref))


def test_full_prefill_is_causal(tiny):
    ids = qd.token_ids(30, qd.TINY.vocab, stream=98)
    a = O.full_prefill(tiny, ids)
    ids2 = ids.copy()
    ids2[-1] = (ids2[-1] + 1) % qd.TINY.vocab
    b = O.full_prefill(tiny, ids2)
    np.testing.assert_allclose(a["K"][:, :-1], b["K"][:, :-1], atol=1e-6)
    np.testing.assert_allclose(a["V"][:, :-1], b["V"][:, :-1], atol=1e-6)


# ----------------------------------------------------------------- fusion special cases

def test_prefix_caching_equals_full_recompute_on_first_chunk(tiny):
    chunks, start, q = tiny_request()
    full = O.full_prefill(tiny, np.concatenate(chunks + [q]))
    c0 = O.chunk_precompute(tiny, chunks[0], store_bf16=False)
    L0 = len(chunks[0])
    np.testing.assert_allclose(c0["K"], full["K"][:, :L0], atol=2e-5)
    np.testing.assert_allclose(c0["V"], full["V"][:, :L0], atol=2e-5)


def test_layer0_reposition_equals_key_at_absolute_offset(tiny):
    chunks, start, q = tiny_request()
    c = 2
    stored = O.chunk_precompute(tiny, chunks[c], store_bf16=False)["K"][0]
    moved = O.rope_reposition(stored, start[c], qd.TINY.theta)
    at_offset = O.full_prefill(tiny, chunks[c], positions=start[c] + np.arange(len(chunks[c])))["K"][0]
    np.testing.assert_allclose(moved, at_offset, atol=2e-5)


def test_ratio_one_equals_full_recompute(tiny):
    chunks, start, q = tiny_request()
    kv = [O.chunk_precompute(tiny, c, store_bf16=False) for c in chunks]
    ctx = np.concatenate(chunks)
    fused = O.fused_prefill(tiny, kv, ctx, start, q, crit=1, ratio_bp=10000, n_anchor=2)
    full = O.full_prefill(tiny, np.concatenate([ctx, q]))
    assert len(fused["sel"]) == len(ctx)
    np.testing.assert_allclose(fused["K"], full["K"], atol=5e-5)
    np.testing.assert_allclose(fused["V"], full["V"], atol=5e-5)
    np.testing.assert_allclose(fused["logits"], full["logits"], atol=1e-4)


def test_single_chunk_ratio_zero_is_prefix_caching(tiny):
    chunks, start, q = tiny_request(n_chunks=1)
    kv = [O.chunk_precompute(tiny, chunks[0], store_bf16=False)]
    fused = O.fused_prefill(tiny, kv, chunks[0], start, q, crit=1, ratio_bp=0, n_anchor=2)
    full = O.full_prefill(tiny, np.concatenate([chunks[0], q]))
    assert len(fused["sel"]) == 0
    np.testing.assert_allclose(fused["K"], full["K"], atol=5e-5)
    np.testing.assert_allclose(fused["logits"], full["logits"], atol=1e-4)


def test_ratio_zero_is_full_kv_reuse(tiny):
    chunks, start, q = tiny_request()
    kv = [O.chunk_precompute(tiny, c) for c in chunks]
    fused = O.fused_prefill(tiny, kv, np.concatenate(chunks), start, q, crit=1, ratio_bp=0, n_anchor=2)
    C = int(start[-1])
    for l in range(qd.TINY.n_layers):
        for c in range(3):
            np.testing.assert_array_equal(fused["V"][l][start[c]:start[c + 1]], kv[c]["V"][l])
            np.testing.assert_allclose(fused["K"][l][start[c]:start[c + 1]],
                                       O.rope_reposition(kv[c]["K"][l], start[c], qd.TINY.theta), atol=0)
    assert list(fused["rows"]) == list(range(C, C + len(q)))


def test_probe_with_every_token_as_anchor_is_the_real_query(tiny):
    # One chunk at offset 0 whose anchors are all its tokens: the probe is an exact prefix-cached prefill.
    chunks, start, q = tiny_request(n_chunks=1)
    kv = [O.chunk_precompute(tiny, chunks[0], store_bf16=False)]
    fused = O.fused_prefill(tiny, kv, chunks[0], start, q, crit=1, ratio_bp=0, n_anchor=len(chunks[0]))
    full = O.full_prefill(tiny, np.concatenate([chunks[0], q]), capture_q_layer=1)
    np.testing.assert_allclose(fused["q_crit"], full["q"][len(chunks[0]):], atol=5e-5)


def test_probe_without_anchors_is_the_query_alone(tiny):
    chunks, start, q = tiny_request()
    C = int(start[-1])
    qc = O.anchor_probe(tiny, q, [], [], np.zeros(0, np.int64), C, crit=1)
    alone = O.full_prefill(tiny, q, positions=C + np.arange(len(q)), capture_q_layer=1)
    np.testing.assert_allclose(qc, alone["q"], atol=2e-5)


# ----------------------------------------------------------------- scores, selection, anchors

def test_scores_bruteforce_tiny():
    rng = np.random.default_rng(5)
    nq, Hq, Hkv, C, D = 2, 4, 2, 5, 4
    q = rng.standard_normal((nq, Hq, D)).astype(np.float32)
    K = rng.standard_normal((C, Hkv, D)).astype(np.float32)
    want = [0.0] * C
    for r in range(nq):
        for h in range(Hq):
            logits = [0.7 * sum(float(q[r, h, d]) * float(K[j, h // 2, d]) for d in range(D)) for j in range(C)]
            z = sum(math.exp(v) for v in logits)
            for j in range(C):
                want[j] += math.exp(logits[j]) / z
    np.testing.assert_allclose(O.profile_scores(q, K, 0.7), want, rtol=1e-12)


def test_scores_invariants():
    t = qd.sweep_tensors(300, n_query=5, Hq=8, Hkv=2, D=16)
    q, K = O.as_f32(t["Q"]), O.as_f32(t["K"])
    s = O.profile_scores(q, K, 1.0)
    assert abs(s.sum() - 8 * 5) < 1e-9
    flat = np.broadcast_to(K[:1], K.shape).copy()
    np.testing.assert_allclose(O.profile_scores(q, flat, 1.0), 8 * 5 / 300, rtol=1e-12)


def test_num_selected_golden():
    # N = ceil(ratio * |C|), as in Cache-Craft's N = ceil(CFO * |C_i|)
    for line in open(os.path.join(GOLDEN, "num_selected.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        C, bp, N = (int(v) for v in line.split())
        assert O.num_selected(C, bp) == N


def test_topn_bruteforce_with_ties():
    rng = np.random.default_rng(6)
    for C in (1, 7, 64, 1000):
        s = rng.integers(0, 5, C).astype(np.float64) * 0.25   # many exact ties
        for N in sorted({0, 1, C // 3, C - 1, C}):
            N = max(0, N)
            want = sorted(sorted(range(C), key=lambda j: (-s[j], j))[:N])
            assert list(O.topn_select(s, N)) == want


def test_anchors_bruteforce_and_rotation_invariance():
    rng = np.random.default_rng(7)
    K = rng.standard_normal((50, 2, 16)).astype(np.float32)
    K[10] = K[3]            # an exact norm tie: the lower index wins
    start = np.array([0, 20, 50])
    a = O.keynorm_anchors(K, start, 4)
    for c in range(2):
        rows = K[start[c]:start[c + 1]].astype(np.float64)
        norms = [math.sqrt(float(np.sum(r * r))) for r in rows]
        assert list(a[c]) == sorted(sorted(range(len(norms)), key=lambda i: (-norms[i], i))[:4])
    moved = O.rope_reposition(K, np.repeat(start[:-1], np.diff(start)) + 1000, 1e4)
    assert np.array_equal(O.keynorm_anchors(moved, start, 4), a)


def test_sparse_rows_equal_dense_causal_rows():
    rng = np.random.default_rng(8)
    T, Hq, Hkv, D = 90, 4, 2, 16
    q = rng.standard_normal((T, Hq, D)).astype(np.float32)
    K = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    V = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    dense = _sdpa_reference(q, np.arange(T), K, V, 0.5)
    S = np.sort(rng.choice(T, 17, replace=False))
    np.testing.assert_allclose(O.causal_attention(q[S], S, K, V, 0.5), dense[S], atol=1e-6)


def test_round_bf16_matches_library():
    rng = np.random.default_rng(9)
    a = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 100,
                        np.array([1.00390625, 1.01171875, -2.0078125, 0.0, -0.0], np.float32)])
    want = torch.from_numpy(a).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(O.round_bf16(a), want)


# ----------------------------------------------------------------- selector variants (QCLast, QCAll, HKVD)

def _one_chunk_all_anchors(tiny):
    chunks, start, q = tiny_request(n_chunks=1)
    kv = [O.chunk_precompute(tiny, chunks[0], store_bf16=False)]
    return chunks[0], start, q, kv


def test_qclast_probe_is_the_real_query_at_the_last_layer(tiny):
    # crit = L-1 with every token an anchor of the only chunk: q at the last layer is full prefill's q there.
    ctx, start, q, kv = _one_chunk_all_anchors(tiny)
    L = qd.TINY.n_layers
    fused = O.fused_prefill(tiny, kv, ctx, start, q, crit=L - 1, ratio_bp=0, n_anchor=len(ctx))
    full = O.full_prefill(tiny, np.concatenate([ctx, q]), capture_q_layer=L - 1)
    np.testing.assert_allclose(fused["q_crit"], full["q"][len(ctx):], atol=5e-5)


def test_qcall_scores_bruteforce_from_full_prefill(tiny):
    # Same exact-probe setting: QCAll's scores are the sum over layers of each
    # layer's softmax mass on every context key, from full prefill's q and K.
    ctx, start, q, kv = _one_chunk_all_anchors(tiny)
    s = qd.TINY
    C, Qn, G = len(ctx), len(q), s.n_heads // s.n_kv_heads
    fused = O.fused_prefill(tiny, kv, ctx, start, q, crit=1, ratio_bp=0, n_anchor=C, selector="all")
    want = np.zeros(C)
    for l in range(s.n_layers):
        full = O.full_prefill(tiny, np.concatenate([ctx, q]), capture_q_layer=l)
        ql, Kl = full["q"][C:].astype(np.float64), full["K"][l][:C].astype(np.float64)
        for r in range(Qn):
            for h in range(s.n_heads):
                logit = [math.fsum(ql[r, h] * Kl[j, h // G]) / math.sqrt(s.head_dim) for j in range(C)]
                mx = max(logit)
                e = [math.exp(v - mx) for v in logit]
                tot = math.fsum(e)
                for j in range(C):
                    want[j] += e[j] / tot
    np.testing.assert_allclose(fused["scores"], want, rtol=2e-4, atol=1e-6)


def test_qcall_invariants_and_one_layer_reduction():
    s1 = dataclasses.replace(qd.TINY, n_layers=1)
    m1 = O.OracleModel(qd.ModelWeights(s1))
    chunks = [qd.chunk_tokens(c, 32, s1.vocab) for c in range(3)]
    start = np.arange(4) * 32
    q = qd.query_tokens(0, 8, s1.vocab)
    kv = [O.chunk_precompute(m1, c) for c in chunks]
    ctx = np.concatenate(chunks)
    a = O.fused_prefill(m1, kv, ctx, start, q, crit=0, ratio_bp=2000, n_anchor=2, selector="all")
    b = O.fused_prefill(m1, kv, ctx, start, q, crit=0, ratio_bp=2000, n_anchor=2)
    np.testing.assert_allclose(a["scores"], b["scores"], atol=1e-12)   # one layer: all layers == the critical one
    np.testing.assert_array_equal(a["sel"], b["sel"])
    tiny2 = O.OracleModel(qd.ModelWeights(qd.TINY))
    kv2 = [O.chunk_precompute(tiny2, c) for c in chunks]
    c2 = O.fused_prefill(tiny2, kv2, ctx, start, q, crit=1, ratio_bp=2000, n_anchor=2, selector="all")
    # every layer's softmax puts mass 1 per (query row, head) on the context keys
    assert abs(c2["scores"].sum() - qd.TINY.n_layers * len(q) * qd.TINY.n_heads) < 1e-9 * c2["scores"].sum()


def test_hkvd_full_ratio_is_full_recompute(tiny):
    chunks, start, q = tiny_request()
    kv = [O.chunk_precompute(tiny, c, store_bf16=False) for c in chunks]
    ctx = np.concatenate(chunks)
    out = O.hkvd_prefill(tiny, kv, ctx, start, q, [10000] * qd.TINY.n_layers)
    full = O.full_prefill(tiny, np.concatenate([ctx, q]))
    np.testing.assert_allclose(out["K"], full["K"], atol=5e-5)
    np.testing.assert_allclose(out["V"], full["V"], atol=5e-5)
    np.testing.assert_allclose(out["logits"], full["logits"], atol=1e-4)


def test_hkvd_zero_ratio_is_full_kv_reuse(tiny):
    chunks, start, q = tiny_request()
    kv = [O.chunk_precompute(tiny, c) for c in chunks]
    ctx = np.concatenate(chunks)
    out = O.hkvd_prefill(tiny, kv, ctx, start, q, [0] * qd.TINY.n_layers)
    reuse = O.fused_prefill(tiny, kv, ctx, start, q, crit=1, ratio_bp=0, n_anchor=2)
    assert all(len(sl) == 0 for sl in out["layer_sel"])
    np.testing.assert_array_equal(out["K"], reuse["K"])
    np.testing.assert_allclose(out["logits"], reuse["logits"], atol=1e-9)


def _dev_bruteforce(K_fresh, V_fresh, K_reused, V_reused, rows):
    out = []
    for j in rows:
        acc = 0.0
        for h in range(K_fresh.shape[1]):
            for e in range(K_fresh.shape[2]):
                dk = float(K_fresh[j, h, e]) - float(K_reused[j, h, e])
                dv = float(V_fresh[j, h, e]) - float(V_reused[j, h, e])
                acc += dk * dk + dv * dv
        out.append(acc)
    return np.array(out)


def test_hkvd_deviation_bruteforce_from_full_prefill(tiny):
    # At layer 0 the fresh K/V of every context token is full prefill's layer-0 K/V; with
    # layer 0 keeping every token, layer 1's fresh K/V is full prefill's layer-1 K/V too.
    chunks, start, q = tiny_request()
    kv = [O.chunk_precompute(tiny, c) for c in chunks]
    ctx = np.concatenate(chunks)
    C = len(ctx)
    full = O.full_prefill(tiny, np.concatenate([ctx, q]))
    out = O.hkvd_prefill(tiny, kv, ctx, start, q, [10000, 3000])
    row_delta = np.repeat(start[:-1], np.diff(start))
    for l in (0, 1):
        Kr = O.rope_reposition(np.concatenate([c["K"][l] for c in kv]), row_delta, qd.TINY.theta)
        Vr = np.concatenate([c["V"][l] for c in kv])
        want = _dev_bruteforce(full["K"][l], full["V"][l], Kr, Vr, range(C))
        np.testing.assert_allclose(out["layer_dev"][l], want, rtol=1e-4, atol=1e-7)
    order = sorted(range(C), key=lambda j: (-want[j], j))   # layer 1: top 30% by deviation, ties low index
    assert list(out["layer_sel"][1]) == sorted(order[:O.num_selected(C, 3000)])


def test_hkvd_gradual_filtering_nests(tiny):
    chunks, start, q = tiny_request()
    kv = [O.chunk_precompute(tiny, c) for c in chunks]
    ctx = np.concatenate(chunks)
    C = len(ctx)
    out = O.hkvd_prefill(tiny, kv, ctx, start, q, [5000, 2000])
    a, b = out["layer_sel"]
    assert len(a) == O.num_selected(C, 5000) and len(b) == O.num_selected(C, 2000)
    assert np.all(np.diff(a) > 0) and np.all(np.diff(b) > 0) and set(b) <= set(a)
    assert len(out["layer_dev"][1]) == len(a)   # layer 1 measures only the rows kept after layer 0


# ----------------------------------------------------------------- offsets in the probe and in profiling

def test_multichunk_probe_and_scores_use_absolute_positions(tiny):
    # Three chunks, critical layer 1, every token an anchor.  Layer-0 K depends only on the
    # token and its position and layer-0 V only on the token, so the anchors' re-rotated
    # layer-0 K/V are full prefill's, and the probe's q at layer 1 is full prefill's q of the
    # query rows.  A probe that dropped (or negated) the chunks' offsets would see keys at the
    # wrong positions and fail here; the single-chunk pins above cannot see that.
    chunks, start, q = tiny_request()
    C = int(start[-1])
    kv = [O.chunk_precompute(tiny, c, store_bf16=False) for c in chunks]
    ctx = np.concatenate(chunks)
    fused = O.fused_prefill(tiny, kv, ctx, start, q, crit=1, ratio_bp=1500, n_anchor=len(chunks[0]))
    full = O.full_prefill(tiny, np.concatenate([ctx, q]), capture_q_layer=1)
    np.testing.assert_allclose(fused["q_crit"], full["q"][C:], atol=5e-5)
    # The scores: each chunk prefilled alone at its absolute positions gives its layer-1 keys
    # where the fused layout puts them (attention inside a chunk sees only relative
    # positions); softmax of q_crit over them, summed by explicit loops.
    s = qd.TINY
    G = s.n_heads // s.n_kv_heads
    K1 = np.concatenate([O.full_prefill(tiny, chunks[c], positions=start[c] + np.arange(len(chunks[c])))["K"][1]
                         for c in range(len(chunks))]).astype(np.float64)
    qc = fused["q_crit"].astype(np.float64)
    want = np.zeros(C)
    for r in range(len(q)):
        for h in range(s.n_heads):
            logit = [math.fsum(qc[r, h] * K1[j, h // G]) / math.sqrt(s.head_dim) for j in range(C)]
            mx = max(logit)
            e = [math.exp(v - mx) for v in logit]
            tot = math.fsum(e)
            for j in range(C):
                want[j] += e[j] / tot
    np.testing.assert_allclose(fused["scores"], want, rtol=1e-4, atol=1e-7)
