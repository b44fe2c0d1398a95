"""Model-level parity of the CUDA path with the CPU oracle (GPU).

* one decoder layer (qcf_fused_layer_forward) at the tiny and the 8B layer shape;
* full prefill of the tiny model (qcf_full_prefill);
* the whole fused prefill of the tiny request, free-running and with the
  oracle's selection forced (so a discrete flip cannot cascade), plus the
  ratio-1 and ratio-0 special cases;
* the 8B-shaped request at full size: properties that hold at any size and
  sampled rows the oracle computes one by one.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import qcfdata as qd
from oracle import qcf_oracle as O
from _parity import assert_close, assert_same_selection

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = dict(atol=2e-2, rtol=2e-2, rms_scaled=True)   # bf16 hidden states and K/V


@pytest.fixture(scope="module")
def M():
    from rag_kv_cache_re_gb300 import model
    return model


@pytest.fixture(scope="module")
def Q():
    from rag_kv_cache_re_gb300 import qcf
    return qcf


def f32(t):
    return t.float().cpu().numpy()


def _layer_case(M, Q, spec, n_sel, T, Cx, seed):
    weights = qd.ModelWeights(spec)
    dm = M.DeviceModel(weights, DEV, max_pos=T + 8)
    om = O.OracleModel(weights)
    rows = np.concatenate([qd.selected_indices(Cx, n_sel, "uniform"), np.arange(Cx, T)]).astype(np.int32)
    n = len(rows)
    x = torch.randn((n, spec.d_model), generator=torch.Generator().manual_seed(seed)).float()
    Kc = qd.normal_bf16((T, spec.n_kv_heads, spec.head_dim), 1.0, seed + 1)
    Vc = qd.normal_bf16((T, spec.n_kv_heads, spec.head_dim), 1.0, seed + 2)
    xg, Kg, Vg = x.to(DEV), Kc.to(DEV), Vc.to(DEV)
    r = torch.from_numpy(rows).to(DEV)
    Q.qcf_fused_layer_forward(dm, 0, xg, r, r, Kg, Vg)
    torch.cuda.synchronize()
    Ko, Vo = f32(Kc), f32(Vc)
    xr = O.layer_forward(x.numpy(), om.layer(0), spec, rows, rows, Ko, Vo)
    assert_close(xg.cpu().numpy(), xr, what="x after the layer", **TOL)
    assert_close(f32(Kg)[rows], Ko[rows], what="fresh K", **TOL)
    assert_close(f32(Vg)[rows], Vo[rows], what="fresh V", **TOL)
    keep = np.setdiff1d(np.arange(T), rows)
    assert torch.equal(Kg.cpu()[keep], Kc[keep]) and torch.equal(Vg.cpu()[keep], Vc[keep])
    assert Q.qcf_query_status() == 0


def test_layer_forward_tiny(M, Q):
    _layer_case(M, Q, qd.TINY, n_sel=15, T=104, Cx=96, seed=41)


def test_layer_forward_8b_layer_shape(M, Q):
    spec = dataclasses.replace(qd.LLAMA8B, n_layers=1, vocab=512)
    _layer_case(M, Q, spec, n_sel=768, T=5184, Cx=5120, seed=42)


def test_layer_forward_8b_two_row_tiles(M, Q):
    # 144 rows: two 128-row GEMM tiles, the second holding 16 rows
    spec = dataclasses.replace(qd.LLAMA8B, n_layers=1, vocab=512)
    _layer_case(M, Q, spec, n_sel=80, T=5184, Cx=5120, seed=43)


def test_full_prefill_tiny(M, Q):
    weights = qd.ModelWeights(qd.TINY)
    dm = M.DeviceModel(weights, DEV, max_pos=256)
    om = O.OracleModel(weights)
    ids = qd.token_ids(104, qd.TINY.vocab, stream=7)
    K, V, logits, tok = Q.qcf_full_prefill(dm, torch.from_numpy(ids).to(DEV))
    torch.cuda.synchronize()
    ref = O.full_prefill(om, ids)
    for l in range(qd.TINY.n_layers):
        assert_close(f32(K[l]), ref["K"][l], what=f"K layer {l}", **TOL)
        assert_close(f32(V[l]), ref["V"][l], what=f"V layer {l}", **TOL)
    assert_close(logits.cpu().numpy(), ref["logits"], what="logits", **TOL)
    top2 = np.sort(ref["logits"])[-2:]
    if top2[1] - top2[0] > 4e-2 * (1 + abs(top2[1])):
        assert int(tok.item()) == ref["token"]


# ----------------------------------------------------------------- the tiny request end to end

@pytest.fixture(scope="module")
def tiny_world(M):
    spec, req = qd.TINY, qd.TINY_REQ
    weights = qd.ModelWeights(spec)
    dm = M.DeviceModel(weights, DEV, max_pos=256)
    om = O.OracleModel(weights)
    ids = list(range(req.n_chunks))
    toks = [qd.chunk_tokens(c, req.chunk_len, spec.vocab) for c in ids]
    kv = [O.chunk_precompute(om, t) for t in toks]          # stored as bf16
    store = M.ChunkStore(dm, req.crit_layer, req.n_anchor)
    for c, t, k in zip(ids, toks, kv):
        store.add_precomputed(c, t, torch.from_numpy(k["K"]).to(torch.bfloat16), torch.from_numpy(k["V"]).to(torch.bfloat16))
    query = qd.query_tokens(0, req.query_len, spec.vocab)
    start = np.arange(req.n_chunks + 1) * req.chunk_len
    return dict(spec=spec, req=req, dm=dm, om=om, ids=ids, toks=toks, kv=kv, store=store, query=query, start=start)


def _oracle_fused(w, ratio_bp, forced=None):
    return O.fused_prefill(w["om"], w["kv"], np.concatenate(w["toks"]), w["start"], w["query"], w["req"].crit_layer,
                           ratio_bp, w["req"].n_anchor, forced_sel=forced)


def _check_fused(w, fr, ref):
    spec = w["spec"]
    for l in range(spec.n_layers):
        assert_close(f32(fr.K[l]), ref["K"][l], what=f"fused K layer {l}", **TOL)
        assert_close(f32(fr.V[l]), ref["V"][l], what=f"fused V layer {l}", **TOL)
    assert_close(fr.x_rows.cpu().numpy(), ref["x"], what="recomputed rows", **TOL)
    assert_close(fr.logits.cpu().numpy(), ref["logits"], what="logits", **TOL)
    top2 = np.sort(ref["logits"])[-2:]
    if top2[1] - top2[0] > 4e-2 * (1 + abs(top2[1])):
        assert int(fr.token.item()) == ref["token"] == int(fr.token_host.item())


def _streams(two):
    """One stream (copies and compute in order) or two (the layer copies and re-rotations on
    a copy stream, ordered against the compute stream by events only)."""
    return (torch.cuda.Stream(), torch.cuda.Stream()) if two else (None, None)


@pytest.mark.parametrize("two_streams", [False, True], ids=["one_stream", "two_streams"])
def test_tiny_request_anchors_and_probe(M, Q, tiny_world, two_streams):
    w = tiny_world
    ref = _oracle_fused(w, w["req"].ratio_bp)
    for c in w["ids"]:
        Kc = w["kv"][c]["K"][w["req"].crit_layer].astype(np.float64)
        nrm = np.sqrt(np.sum(Kc.reshape(Kc.shape[0], -1) ** 2, axis=1))
        assert_same_selection(w["store"].chunks[c].anchor_idx, nrm, w["req"].n_anchor, 1e-5 * nrm.max(), "anchors")
    fr = M.FusedRequest(w["dm"], w["store"], w["ids"], w["query"], w["req"].ratio_bp)
    fr.run(*_streams(two_streams))
    torch.cuda.synchronize()
    assert Q.qcf_query_status() == 0
    assert_close(f32(fr.q_crit), ref["q_crit"], what="q_crit", **TOL)
    sc = fr.scores.cpu().numpy()
    assert_close(sc, ref["scores"], atol=2e-2, rtol=2e-2, what="scores")
    assert abs(sc.sum() - w["spec"].n_heads * len(w["query"])) < 1e-3 * sc.sum()
    # the selection may only differ between tokens whose oracle scores are closer than the score error
    tie = 2e-2 * (1 + np.abs(ref["scores"]).max())
    assert_same_selection(fr.selected.cpu().numpy(), ref["scores"], ref["N"], tie, "selection")
    got_sel = np.sort(fr.selected.cpu().numpy())
    if np.array_equal(got_sel, ref["sel"]):
        _check_fused(w, fr, ref)


@pytest.mark.parametrize("two_streams", [False, True], ids=["one_stream", "two_streams"])
def test_tiny_request_forced_selection(M, Q, tiny_world, two_streams):
    w = tiny_world
    ref = _oracle_fused(w, w["req"].ratio_bp)
    fr = M.FusedRequest(w["dm"], w["store"], w["ids"], w["query"], w["req"].ratio_bp, forced_sel=ref["sel"])
    fr.run(*_streams(two_streams), ids_from_host=True)
    torch.cuda.synchronize()
    assert np.array_equal(np.sort(fr.selected.cpu().numpy()), ref["sel"])
    _check_fused(w, fr, ref)


@pytest.mark.parametrize("two_streams", [False, True], ids=["one_stream", "two_streams"])
@pytest.mark.parametrize("ratio_bp", [0, 10000])
def test_tiny_request_special_ratios(M, Q, tiny_world, ratio_bp, two_streams):
    w = tiny_world
    ref = _oracle_fused(w, ratio_bp)
    fr = M.FusedRequest(w["dm"], w["store"], w["ids"], w["query"], ratio_bp)
    fr.run(*_streams(two_streams))
    torch.cuda.synchronize()
    assert fr.N == ref["N"]
    _check_fused(w, fr, ref)
    if ratio_bp == 10000:   # every row recomputed: the fused path is the GPU full prefill
        K, V, logits, _ = Q.qcf_full_prefill(w["dm"], fr.ids)
        torch.cuda.synchronize()
        for l in range(w["spec"].n_layers):
            assert_close(f32(fr.K[l]), f32(K[l]), atol=1e-2, rtol=1e-2, what="ratio 1 vs full prefill")


# ----------------------------------------------------------------- the 8B-shaped request at full size

def test_llama8b_request_full_size(M, Q):
    spec, req = qd.LLAMA8B, qd.LLAMA8B_REQ
    weights = qd.ModelWeights(spec, device=DEV)
    dm = M.DeviceModel(weights, DEV, max_pos=8192)
    del weights
    store = M.ChunkStore(dm, req.crit_layer, req.n_anchor)
    ids = list(range(req.n_chunks))
    for c in ids:
        K = torch.stack([qd.synthetic_chunk_kv(spec, c, req.chunk_len, l, device=DEV)["K"] for l in range(spec.n_layers)])
        V = torch.stack([qd.synthetic_chunk_kv(spec, c, req.chunk_len, l, device=DEV)["V"] for l in range(spec.n_layers)])
        store.add_precomputed(c, qd.chunk_tokens(c, req.chunk_len, spec.vocab), K, V)
    query = qd.query_tokens(0, req.query_len, spec.vocab)
    fr = M.FusedRequest(dm, store, ids, query, req.ratio_bp)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    fr.run(cs, xs)
    torch.cuda.synchronize()
    assert Q.qcf_query_status() == 0
    C, T, N = fr.C, fr.T, fr.N
    assert (C, N) == (5120, 768)
    sel = fr.selected.cpu().numpy()
    assert np.all(np.diff(sel) > 0) and sel[0] >= 0 and sel[-1] < C
    sc = fr.scores.double().cpu().numpy()
    assert np.all(sc >= 0) and abs(sc.sum() - spec.n_heads * req.query_len) < 1e-3 * sc.sum()
    # the selection is exactly the top-N of the kernel's own scores
    assert np.array_equal(sel, O.topn_select(fr.scores.cpu().numpy().astype(np.float64), N))
    lg = fr.logits.cpu().numpy()
    assert np.all(np.isfinite(lg)) and int(fr.token_host.item()) == int(np.argmax(lg))
    # unselected context rows keep the stored values, keys re-rotated to their offsets
    rng = np.random.default_rng(0)
    unsel = np.setdiff1d(np.arange(C), sel)
    for l in (0, req.crit_layer, spec.n_layers - 1):
        rows = np.sort(rng.choice(unsel, 64, replace=False))
        for r in rows[:16]:
            c, i = divmod(int(r), req.chunk_len)
            stored = store.chunks[c]
            np.testing.assert_array_equal(f32(fr.V[l][r]), f32(stored.V[l][i]))
            want = O.rope_reposition(f32(stored.K[l][i:i + 1]), c * req.chunk_len, spec.theta)[0]
            assert_close(f32(fr.K[l][r]), want, atol=1e-6, rtol=2.0 ** -8, what=f"reused K layer {l}")
        # recomputed rows hold fresh keys (not the stored ones)
        r = int(sel[len(sel) // 2])
        c, i = divmod(r, req.chunk_len)
        want = O.rope_reposition(f32(store.chunks[c].K[l][i:i + 1]), c * req.chunk_len, spec.theta)[0]
        assert np.max(np.abs(f32(fr.K[l][r]) - want)) > 1e-2
