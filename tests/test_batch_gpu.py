"""Batched requests that share retrieved chunks (GPU).

Each distinct chunk's K/V of a layer crosses the host link once and is written into
every request's fused cache with that request's own offset (QCFuse 1: chunks of
different queries overlap by more than 70 %; 2.B: content-keyed cache index).  The
batch must give every request exactly what qcf_request_prefill gives it alone, and
send only the distinct chunks' bytes.
"""
import numpy as np
import pytest
import torch

import qcfdata as qd
from oracle import qcf_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def M():
    from rag_kv_cache_re_gb300 import model
    return model


@pytest.fixture(scope="module")
def world(M):
    spec, req = qd.TINY, qd.TINY_REQ
    weights = qd.ModelWeights(spec)
    dm = M.DeviceModel(weights, DEV, max_pos=256)
    om = O.OracleModel(weights)
    store = M.ChunkStore(dm, req.crit_layer, req.n_anchor)
    kv = {}
    for c in range(4):
        t = qd.chunk_tokens(c, req.chunk_len, spec.vocab)
        k = kv[c] = O.chunk_precompute(om, t)
        store.add_precomputed(c, t, torch.from_numpy(k["K"]).to(torch.bfloat16), torch.from_numpy(k["V"]).to(torch.bfloat16))
    # chunk id 10 carries chunk 1's tokens: the content-keyed store maps it to the same stored chunk
    store.add_precomputed(10, qd.chunk_tokens(1, req.chunk_len, spec.vocab),
                          torch.zeros((spec.n_layers, req.chunk_len, spec.n_kv_heads, spec.head_dim), dtype=torch.bfloat16),
                          torch.zeros((spec.n_layers, req.chunk_len, spec.n_kv_heads, spec.head_dim), dtype=torch.bfloat16))
    assert store.chunks[10] is store.chunks[1]
    kv[10] = kv[1]
    return dict(spec=spec, req=req, dm=dm, store=store, om=om, kv=kv)


def _requests(M, w, kinds):
    spec, req = w["spec"], w["req"]
    chunk_sets = [[0, 1, 2], [2, 10, 3], [3, 0, 1]]
    out = []
    for i, kind in enumerate(kinds):
        q = qd.query_tokens(i, req.query_len, spec.vocab)
        if kind == "hkvd":
            sched = [3000, req.ratio_bp]
            out.append(M.FusedRequest(w["dm"], w["store"], chunk_sets[i], q, req.ratio_bp, selector=M.SELECT_HKVD,
                                      layer_ratio_bp=sched))
        elif kind == "all":
            out.append(M.FusedRequest(w["dm"], w["store"], chunk_sets[i], q, req.ratio_bp, selector=M.SELECT_ALL_LAYERS))
        else:
            out.append(M.FusedRequest(w["dm"], w["store"], chunk_sets[i], q, req.ratio_bp))
    return out


def _snapshot(fr):
    return {"K": [k.clone() for k in fr.K], "V": [v.clone() for v in fr.V], "sel": fr.selected.clone(),
            "scores": fr.scores.clone(), "logits": fr.logits.clone(), "x": fr.x_rows.clone(), "token": int(fr.token.item())}


@pytest.mark.parametrize("kinds", [("critical", "critical"), ("critical", "hkvd", "all")])
def test_batch_equals_requests_alone(M, world, kinds):
    w = world
    alone = _requests(M, w, kinds)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    for fr in alone:
        fr.run(cs, xs)
    torch.cuda.synchronize()
    ref = [_snapshot(fr) for fr in alone]
    batch = _requests(M, w, kinds)
    h2d = M.run_batch(batch, cs, xs)
    torch.cuda.synchronize()
    for i, (fr, r) in enumerate(zip(batch, ref)):
        for l in range(w["spec"].n_layers):
            assert torch.equal(fr.K[l], r["K"][l]), f"request {i} K layer {l}"
            assert torch.equal(fr.V[l], r["V"][l]), f"request {i} V layer {l}"
        assert torch.equal(fr.selected, r["sel"]) and torch.equal(fr.scores, r["scores"])
        assert torch.equal(fr.logits, r["logits"]) and torch.equal(fr.x_rows, r["x"])
        assert int(fr.token.item()) == r["token"]
    # the distinct chunks' K/V once per layer, one more K copy per distinct critical layer,
    # plus the anchors and two int32 row maps per request
    spec, req = w["spec"], w["req"]
    ids = [[0, 1, 2], [2, 10, 3], [3, 0, 1]][: len(kinds)]
    distinct = {id(w["store"].chunks[c]) for s in ids for c in s}
    row_bytes = spec.n_kv_heads * spec.head_dim * 2
    chunk_layer = req.chunk_len * row_bytes
    crits = {fr.store.crit if fr.selector == M.SELECT_CRITICAL else (spec.n_layers - 1 if fr.selector == M.SELECT_ALL_LAYERS else 0)
             for fr in batch}
    need_k_layers = sum(1 for l in range(spec.n_layers) if any(l != c for c in crits)) if len(crits) > 1 else spec.n_layers - 1
    want = len(distinct) * chunk_layer * (spec.n_layers + need_k_layers + len(crits))
    for fr in batch:
        probe = 0 if fr.selector == M.SELECT_HKVD else (spec.n_layers - 1 if fr.selector == M.SELECT_ALL_LAYERS else fr.store.crit)
        want += 2 * 3 * probe * req.n_anchor * row_bytes + 2 * fr.C * 4
    assert h2d == want
    sequential = sum(len(s) for s in ids) * chunk_layer * 2 * spec.n_layers
    assert h2d < sequential


def test_batch_matches_the_oracle_per_request(M, world):
    """Each request of a batch against the oracle's fused prefill of that request alone, with
    the shared chunks at different offsets in the two requests (chunk 2 is third in one and
    first in the other; chunk id 10 is chunk 1's content in second place).  Selections are
    the oracle's, forced, so every output can be compared element by element."""
    from _parity import assert_close
    w = world
    spec, req = w["spec"], w["req"]
    sets = [[0, 1, 2], [2, 10, 3]]
    refs, batch = [], []
    for i, ids in enumerate(sets):
        q = qd.query_tokens(i, req.query_len, spec.vocab)
        toks = np.concatenate([qd.chunk_tokens(1 if c == 10 else c, req.chunk_len, spec.vocab) for c in ids])
        start = np.arange(len(ids) + 1) * req.chunk_len
        ref = O.fused_prefill(w["om"], [w["kv"][c] for c in ids], toks, start, q, req.crit_layer, req.ratio_bp,
                              req.n_anchor)
        refs.append(ref)
        batch.append(M.FusedRequest(w["dm"], w["store"], ids, q, req.ratio_bp, forced_sel=ref["sel"]))
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    M.run_batch(batch, cs, xs)
    torch.cuda.synchronize()
    tol = dict(atol=2e-2, rtol=2e-2, rms_scaled=True)
    for i, (fr, ref) in enumerate(zip(batch, refs)):
        assert np.array_equal(np.sort(fr.selected.cpu().numpy()), ref["sel"])
        assert_close(fr.q_crit.float().cpu().numpy(), ref["q_crit"], what=f"request {i} q_crit", **tol)
        assert_close(fr.scores.cpu().numpy(), ref["scores"], atol=2e-2, rtol=2e-2, what=f"request {i} scores")
        for l in range(spec.n_layers):
            assert_close(fr.K[l].float().cpu().numpy(), ref["K"][l], what=f"request {i} K layer {l}", **tol)
            assert_close(fr.V[l].float().cpu().numpy(), ref["V"][l], what=f"request {i} V layer {l}", **tol)
        assert_close(fr.x_rows.cpu().numpy(), ref["x"], what=f"request {i} recomputed rows", **tol)
        assert_close(fr.logits.cpu().numpy(), ref["logits"], what=f"request {i} logits", **tol)
