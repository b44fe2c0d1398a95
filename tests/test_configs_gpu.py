"""Full-size parity on the kernel sweep and the 34B / 70B request shapes (GPU).

At these sizes the oracle cannot run the whole path, so the tests check
properties that hold at any size and outputs the oracle computes one by one:
sampled attention rows, re-rotated reused keys, stored values, the selection
against the kernel's own scores, and the score sum.
"""
import math

import numpy as np
import pytest
import torch

import qcfdata as qd
from oracle import qcf_oracle as O
from _parity import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def f32(t):
    return t.float().cpu().numpy()


# ----------------------------------------------------------------- kernel sweep (config 3)

@pytest.mark.parametrize("C", qd.SWEEP_CONTEXTS)
@pytest.mark.parametrize("frac_bp", qd.SWEEP_FRACTIONS_BP)
@pytest.mark.parametrize("pattern", ["uniform", "clusters"])
def test_sweep_sparse_attention_sampled_rows(C, frac_bp, pattern):
    from rag_kv_cache_re_gb300 import qcf as Q
    Hq, Hkv, D = qd.SWEEP_HEADS
    nq = qd.SWEEP_QUERY
    N = O.num_selected(C, frac_bp)
    T = C + nq
    pos = np.concatenate([qd.selected_indices(C, N, pattern), np.arange(C, T)]).astype(np.int32)
    t = qd.sweep_tensors(T, n_query=len(pos), device=DEV)
    q = t["Q"]
    o = Q.qcf_sparse_causal_attn(q, torch.from_numpy(pos).to(DEV), t["K"], t["V"], 1.0)
    torch.cuda.synchronize()
    n = len(pos)
    sample = sorted({0, 1, n // 3, n // 2, N - 1 if N else 0, N, n - 2, n - 1} & set(range(n)))
    Kf, Vf = f32(t["K"]), f32(t["V"])
    ref = O.causal_attention(f32(q[sample]), pos[sample], Kf, Vf, 1.0, block=2)
    assert_close(f32(o[sample]), ref, atol=2e-2, rtol=2e-2, what=f"attention rows {sample}")
    assert Q.qcf_query_status() == 0


@pytest.mark.parametrize("C", qd.SWEEP_CONTEXTS)
def test_sweep_profile_then_topn(C):
    from rag_kv_cache_re_gb300 import qcf as Q
    t = qd.sweep_tensors(C, device=DEV)
    s = Q.qcf_profile_scores(t["Q"], t["K"], 1.0)
    v = s.cpu().numpy()
    assert abs(v.astype(np.float64).sum() - 32 * 64) < 1e-3 * 32 * 64
    for frac_bp in qd.SWEEP_FRACTIONS_BP:
        N = O.num_selected(C, frac_bp)
        sel = Q.qcf_topn_select(s, N).cpu().numpy()
        assert np.array_equal(sel, O.topn_select(v.astype(np.float64), N)), (C, frac_bp)
    if C <= 16384:   # the oracle's scores at these sizes: the selections agree up to near-ties
        ref = O.profile_scores(f32(t["Q"]), f32(t["K"]), 1.0)
        assert_close(v, ref, atol=1e-3, rtol=1e-3, what="scores")


# ----------------------------------------------------------------- request shapes (configs 4 and 5)

def _build(spec, req, device, chunk_ids):
    from rag_kv_cache_re_gb300 import model as M
    weights = qd.ModelWeights(spec, device=device)
    dm = M.DeviceModel(weights, device, max_pos=1 << 16)
    del weights
    torch.cuda.empty_cache()
    store = M.ChunkStore(dm, req.crit_layer, req.n_anchor)
    for c in sorted(set(int(x) for x in chunk_ids)):
        K = torch.stack([qd.synthetic_chunk_kv(spec, c, req.chunk_len, l, device=device)["K"] for l in range(spec.n_layers)])
        V = torch.stack([qd.synthetic_chunk_kv(spec, c, req.chunk_len, l, device=device)["V"] for l in range(spec.n_layers)])
        store.add_precomputed(c, qd.chunk_tokens(c, req.chunk_len, spec.vocab), K, V)
        del K, V
    return dm, store


def _check_request(fr, store, spec, req, layers, rng):
    from rag_kv_cache_re_gb300 import qcf as Q
    C, N = fr.C, fr.N
    assert N == O.num_selected(C, fr.req.ratio_bp)
    sel = fr.selected.cpu().numpy()
    assert len(sel) == N and np.all(np.diff(sel) > 0) and sel[0] >= 0 and sel[-1] < C
    sc = fr.scores.double().cpu().numpy()
    assert np.all(sc >= 0) and abs(sc.sum() - spec.n_heads * fr.Q) < 1e-3 * sc.sum()
    assert np.array_equal(sel, O.topn_select(fr.scores.cpu().numpy().astype(np.float64), N))
    lg = fr.logits.cpu().numpy()
    assert np.all(np.isfinite(lg)) and int(fr.token_host.item()) == int(np.argmax(lg))
    unsel = np.setdiff1d(np.arange(C), sel)
    ids = [int(c) for c in fr.chunk_ids]
    for l in layers:
        for r in np.sort(rng.choice(unsel, 12, replace=False)):
            k, i = divmod(int(r), req.chunk_len)
            stored = store.chunks[ids[k]]
            np.testing.assert_array_equal(f32(fr.V[l][r]), f32(stored.V[l][i]))
            want = O.rope_reposition(f32(stored.K[l][i:i + 1]), k * req.chunk_len, spec.theta)[0]
            assert_close(f32(fr.K[l][r]), want, atol=1e-6, rtol=2.0 ** -8, what=f"reused K layer {l}")
    assert Q.qcf_query_status() == 0


@pytest.mark.parametrize("ratio_bp", [1000, 2000])
def test_yi34b_request_full_size(ratio_bp):
    from rag_kv_cache_re_gb300 import model as M
    spec, req = qd.YI34B, qd.YI34B_REQ
    chunk_ids = list(range(req.n_chunks))
    dm, store = _build(spec, req, DEV, chunk_ids)
    fr = M.FusedRequest(dm, store, chunk_ids, qd.query_tokens(0, req.query_len, spec.vocab), ratio_bp)
    fr.run(torch.cuda.Stream(), torch.cuda.Stream())
    torch.cuda.synchronize()
    assert (fr.C, fr.N) == (20480, 2048 if ratio_bp == 1000 else 4096)
    _check_request(fr, store, spec, req, (0, req.crit_layer, spec.n_layers - 1), np.random.default_rng(1))


def test_llama70b_two_requests_sharing_chunks():
    from rag_kv_cache_re_gb300 import model as M
    spec, req = qd.LLAMA70B, qd.LLAMA70B_REQ
    reqs = qd.shared_chunk_requests(req.n_chunks, 0.70)
    assert len(set(reqs[0]) & set(reqs[1])) == 25
    dm, store = _build(spec, req, DEV, np.concatenate(reqs))
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    frs = []
    for i, ids in enumerate(reqs):   # the batch of two: enqueued back to back, first tokens when both land
        fr = M.FusedRequest(dm, store, ids, qd.query_tokens(i, req.query_len, spec.vocab), req.ratio_bp)
        fr.run(cs, xs)
        frs.append(fr)
    torch.cuda.synchronize()
    rng = np.random.default_rng(2)
    for fr in frs:
        assert (fr.C, fr.N) == (17920, 2688)
        _check_request(fr, store, spec, req, (0, req.crit_layer, spec.n_layers - 1), rng)
    # a chunk shared by both requests sits at different offsets: where neither request
    # recomputed a token, its value rows are equal and each key is the stored key
    # rotated to that request's offset
    # the same two requests as one batch: shared chunks cross the host link once per layer,
    # and every result is bitwise what the request gave alone
    batch = [M.FusedRequest(dm, store, ids, qd.query_tokens(i, req.query_len, spec.vocab), req.ratio_bp)
             for i, ids in enumerate(reqs)]
    h2d = M.run_batch(batch, cs, xs)
    torch.cuda.synchronize()
    for fr, bt in zip(frs, batch):
        assert torch.equal(fr.selected, bt.selected) and torch.equal(fr.logits, bt.logits)
        for l in (0, req.crit_layer, spec.n_layers - 1):
            assert torch.equal(fr.K[l], bt.K[l]) and torch.equal(fr.V[l], bt.V[l])
    row_bytes = spec.n_kv_heads * spec.head_dim * 2
    layer_bytes = req.chunk_len * row_bytes
    n_distinct = len(set(np.concatenate(reqs).tolist()))
    assert n_distinct == 45
    # distinct chunks: V of every layer, K of every other layer, the critical layer's K once;
    # per request: the anchors of the probe layers and two int32 row maps
    per_req = 2 * req.n_chunks * req.crit_layer * req.n_anchor * row_bytes + 2 * req.n_chunks * req.chunk_len * 4
    assert h2d == n_distinct * layer_bytes * 2 * spec.n_layers + 2 * per_req
    assert h2d < 0.7 * 2 * req.n_chunks * layer_bytes * 2 * spec.n_layers   # the two requests alone: 70 chunks
    del batch
    a, b = frs
    shared = sorted(set(a.chunk_ids) & set(b.chunk_ids))[:3]
    sa, sb = set(a.selected.cpu().numpy().tolist()), set(b.selected.cpu().numpy().tolist())
    l = spec.n_layers // 2
    for c in shared:
        ka, kb = a.chunk_ids.index(c), b.chunk_ids.index(c)
        stored = store.chunks[c]
        for i in range(0, req.chunk_len, 97):
            ra, rb = ka * req.chunk_len + i, kb * req.chunk_len + i
            if ra in sa or rb in sb:
                continue
            np.testing.assert_array_equal(f32(a.V[l][ra]), f32(b.V[l][rb]))
            for fr, r, k in ((a, ra, ka), (b, rb, kb)):
                want = O.rope_reposition(f32(stored.K[l][i:i + 1]), k * req.chunk_len, spec.theta)[0]
                assert_close(f32(fr.K[l][r]), want, atol=1e-6, rtol=2.0 ** -8, what="shared chunk re-rotation")
