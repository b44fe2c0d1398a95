"""GPU parity of the selector variants the pages compare QCFuse against (GPU).

* QCLast (profiling at the last layer) and QCAll (query-aware profiling at every
  layer), *QCFuse* section 4, on a three-layer tiny model where the last layer is
  not the critical one;
* CacheBlend's KV-deviation selection with gradual filtering (*KVCache reuse 01*
  1.3.2-1.3.4): the deviation kernel alone, the tiny request layer by layer with the
  kernel's own choices replayed in the oracle, the 100 % schedule against full
  prefill, and the 8B-shaped request at full size through properties and sampled
  rows.
"""
import dataclasses

import numpy as np
import pytest
import torch

import qcfdata as qd
from oracle import qcf_oracle as O
from _parity import assert_close, assert_same_selection

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = dict(atol=2e-2, rtol=2e-2, rms_scaled=True)   # bf16 hidden states and K/V
SPEC3 = dataclasses.replace(qd.TINY, n_layers=3)     # QCLast (crit 2) differs from the critical layer 1


def f32(t):
    return t.float().cpu().numpy()


@pytest.fixture(scope="module")
def M():
    from rag_kv_cache_re_gb300 import model
    return model


@pytest.fixture(scope="module")
def Q():
    from rag_kv_cache_re_gb300 import qcf
    return qcf


@pytest.fixture(scope="module")
def world3(M):
    spec, req = SPEC3, qd.TINY_REQ
    weights = qd.ModelWeights(spec)
    dm = M.DeviceModel(weights, DEV, max_pos=256)
    om = O.OracleModel(weights)
    ids = list(range(req.n_chunks))
    toks = [qd.chunk_tokens(c, req.chunk_len, spec.vocab) for c in ids]
    kv = [O.chunk_precompute(om, t) for t in toks]          # stored as bf16
    stores = {}
    for crit in (1, spec.n_layers - 1):
        st = M.ChunkStore(dm, crit, req.n_anchor)
        for c, t, k in zip(ids, toks, kv):
            st.add_precomputed(c, t, torch.from_numpy(k["K"]).to(torch.bfloat16),
                               torch.from_numpy(k["V"]).to(torch.bfloat16))
        stores[crit] = st
    query = qd.query_tokens(0, req.query_len, spec.vocab)
    start = np.arange(req.n_chunks + 1) * req.chunk_len
    return dict(spec=spec, req=req, dm=dm, om=om, ids=ids, toks=toks, kv=kv, stores=stores, query=query,
                start=start, ctx=np.concatenate(toks))


def _check_rows(w, fr, ref):
    for l in range(w["spec"].n_layers):
        assert_close(f32(fr.K[l]), ref["K"][l], what=f"K layer {l}", **TOL)
        assert_close(f32(fr.V[l]), ref["V"][l], what=f"V layer {l}", **TOL)
    assert_close(fr.x_rows.cpu().numpy(), ref["x"], what="recomputed rows", **TOL)
    assert_close(fr.logits.cpu().numpy(), ref["logits"], what="logits", **TOL)


# ----------------------------------------------------------------- KV deviation kernel

@pytest.mark.parametrize("n,T,Hkv,D", [(37, 100, 4, 16), (1, 1, 8, 128), (300, 5184, 8, 128)])
def test_kv_deviation_kernel(Q, n, T, Hkv, D):
    g = torch.Generator().manual_seed(n * 7 + T)
    pos = torch.randperm(T, generator=g)[:n].sort().values.to(torch.int32)
    k = qd.normal_bf16((n, Hkv, D), 1.0, 61, DEV)
    v = qd.normal_bf16((n, Hkv, D), 1.0, 62, DEV)
    K = qd.normal_bf16((T, Hkv, D), 1.0, 63, DEV)
    V = qd.normal_bf16((T, Hkv, D), 1.0, 64, DEV)
    dev = Q.qcf_kv_deviation(k, v, pos.to(DEV), K, V)
    torch.cuda.synchronize()
    p = pos.numpy()
    ref = O.kv_deviation(f32(k), f32(v), f32(K)[p], f32(V)[p])
    # fp32 sums of exact bf16 differences: relative error of order (entries) * 2^-24
    assert_close(dev.cpu().numpy(), ref, atol=1e-6, rtol=2 * Hkv * D * 2.0 ** -24, what="deviation")
    assert Q.qcf_query_status() == 0


def test_kv_deviation_bad_position_flags(Q):
    k = qd.normal_bf16((2, 4, 16), 1.0, 65, DEV)
    K = qd.normal_bf16((8, 4, 16), 1.0, 66, DEV)
    dev = Q.qcf_kv_deviation(k, k, torch.tensor([3, 8], dtype=torch.int32, device=DEV), K, K)
    torch.cuda.synchronize()
    assert float(dev[1]) == 0.0 and float(dev[0]) > 0.0
    assert Q.qcf_query_status() != 0


# ----------------------------------------------------------------- QCLast and QCAll

def _selector_case(M, Q, w, crit, selector, oracle_selector):
    from rag_kv_cache_re_gb300.model import FusedRequest
    spec, req = w["spec"], w["req"]
    ref = O.fused_prefill(w["om"], w["kv"], w["ctx"], w["start"], w["query"], crit, req.ratio_bp, req.n_anchor,
                          selector=oracle_selector)
    fr = FusedRequest(w["dm"], w["stores"][crit], w["ids"], w["query"], req.ratio_bp, selector=selector)
    fr.run()
    torch.cuda.synchronize()
    assert Q.qcf_query_status() == 0
    sc = fr.scores.cpu().numpy()
    assert_close(sc, ref["scores"], atol=2e-2, rtol=2e-2, what="scores")
    layers = spec.n_layers if oracle_selector == "all" else 1
    assert abs(sc.sum() - layers * spec.n_heads * len(w["query"])) < 1e-3 * sc.sum()
    tie = 2e-2 * (1 + np.abs(ref["scores"]).max())
    assert_same_selection(fr.selected.cpu().numpy(), ref["scores"], ref["N"], tie, "selection")
    # with the oracle's selection the whole recompute must agree
    forced = FusedRequest(w["dm"], w["stores"][crit], w["ids"], w["query"], req.ratio_bp, forced_sel=ref["sel"],
                          selector=selector)
    forced.run()
    torch.cuda.synchronize()
    _check_rows(w, forced, ref)
    return fr, ref


def test_qclast_tiny(M, Q, world3):
    w = world3
    fr, ref = _selector_case(M, Q, w, SPEC3.n_layers - 1, M.SELECT_CRITICAL, "critical")
    assert_close(f32(fr.q_crit), ref["q_crit"], what="q at the last layer", **TOL)


def test_qcall_tiny(M, Q, world3):
    _selector_case(M, Q, world3, 1, M.SELECT_ALL_LAYERS, "all")


# ----------------------------------------------------------------- HKVD gradual filtering

def _hkvd_run(M, w, sched):
    fr = M.FusedRequest(w["dm"], w["stores"][1], w["ids"], w["query"], sched[-1], selector=M.SELECT_HKVD,
                        layer_ratio_bp=sched)
    fr.run()
    torch.cuda.synchronize()
    return fr


@pytest.mark.parametrize("sched", [[5000, 3000, 1500], [10000, 2000, 2000], [1000, 1000, 0]])
def test_hkvd_tiny(M, Q, world3, sched):
    w = world3
    C = int(w["start"][-1])
    fr = _hkvd_run(M, w, sched)
    assert Q.qcf_query_status() == 0
    layer_sel = [np.sort(fr.layer_sel[l, :n].cpu().numpy()) for l, n in enumerate(fr.layer_N)]
    for l in range(1, len(sched)):
        assert set(layer_sel[l]) <= set(layer_sel[l - 1]), "gradual filtering must nest"
    # replay the kernel's choices in the oracle; then every layer's choice must be a top-N of
    # the oracle's deviations (up to near ties) and every tensor must agree
    ref = O.hkvd_prefill(w["om"], w["kv"], w["ctx"], w["start"], w["query"], sched, forced_layer_sel=layer_sel)
    for l, n in enumerate(fr.layer_N):
        dev = ref["layer_dev"][l]
        prev = np.arange(C) if l == 0 else layer_sel[l - 1]
        got = np.searchsorted(prev, layer_sel[l])
        assert_same_selection(got, dev, n, 2e-2 * (1 + dev.max()), f"layer {l} selection")
    assert_close(fr.scores.cpu().numpy(), ref["layer_dev"][0], atol=2e-2, rtol=2e-2, rms_scaled=True,
                 what="layer-0 deviation")
    np.testing.assert_array_equal(np.sort(fr.selected.cpu().numpy()), ref["sel"])
    _check_rows(w, fr, ref)


def test_hkvd_full_schedule_is_full_prefill(M, Q, world3):
    w = world3
    fr = _hkvd_run(M, w, [10000] * SPEC3.n_layers)
    K, V, logits, _ = Q.qcf_full_prefill(w["dm"], fr.ids)
    torch.cuda.synchronize()
    for l in range(SPEC3.n_layers):
        assert_close(f32(fr.K[l]), f32(K[l]), atol=1e-2, rtol=1e-2, what="HKVD 100 % vs full prefill")
    assert_close(fr.logits.cpu().numpy(), logits.cpu().numpy(), atol=1e-2, rtol=1e-2, what="logits")


def test_hkvd_llama8b_full_size(M, Q):
    spec, req = qd.LLAMA8B, qd.LLAMA8B_REQ
    weights = qd.ModelWeights(spec, device=DEV)
    dm = M.DeviceModel(weights, DEV, max_pos=8192)
    w0 = {k: weights.layer(0)[k].float().cpu().numpy() for k in ("wk", "wv")}
    store = M.ChunkStore(dm, req.crit_layer, req.n_anchor)
    ids = list(range(req.n_chunks))
    for c in ids:
        K = torch.stack([qd.synthetic_chunk_kv(spec, c, req.chunk_len, l, device=DEV)["K"] for l in range(spec.n_layers)])
        V = torch.stack([qd.synthetic_chunk_kv(spec, c, req.chunk_len, l, device=DEV)["V"] for l in range(spec.n_layers)])
        store.add_precomputed(c, qd.chunk_tokens(c, req.chunk_len, spec.vocab), K, V)
        del K, V
    query = qd.query_tokens(0, req.query_len, spec.vocab)
    L = spec.n_layers
    sched = [int(round(2 * req.ratio_bp - req.ratio_bp * l / (L - 1))) for l in range(L)]   # 2r down to r
    sched[-1] = req.ratio_bp
    fr = M.FusedRequest(dm, store, ids, query, req.ratio_bp, selector=M.SELECT_HKVD, layer_ratio_bp=sched)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    fr.run(cs, xs)
    torch.cuda.synchronize()
    assert Q.qcf_query_status() == 0
    C = fr.C
    sels = [np.sort(fr.layer_sel[l, :n].cpu().numpy()) for l, n in enumerate(fr.layer_N)]
    for l, s in enumerate(sels):
        assert len(s) == O.num_selected(C, sched[l]) and np.all(np.diff(s) > 0) and s[0] >= 0 and s[-1] < C
        if l:
            assert set(s) <= set(sels[l - 1])
    lg = fr.logits.cpu().numpy()
    assert np.all(np.isfinite(lg)) and int(fr.token_host.item()) == int(np.argmax(lg))
    # layer-0 deviation of sampled context rows: fresh K/V from the token's embedding
    dev0 = fr.scores.cpu().numpy()
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(C, 16, replace=False))
    toks = np.concatenate([store.chunks[c].tokens for c in ids])[rows]
    emb = weights.embed()[torch.as_tensor(toks.astype(np.int64), device=DEV)].float().cpu().numpy()
    W0 = {"g_attn": np.ones(spec.d_model, np.float32), **w0}
    k, v = O.kv_projection(emb, W0, spec, rows)
    for i, r in enumerate(rows):
        ci, j = divmod(int(r), req.chunk_len)
        Ks = O.rope_reposition(f32(store.chunks[ids[ci]].K[0][j:j + 1]), ci * req.chunk_len, spec.theta)
        Vs = f32(store.chunks[ids[ci]].V[0][j:j + 1])
        want = O.kv_deviation(k[i:i + 1], v[i:i + 1], Ks, Vs)[0]
        assert abs(dev0[r] - want) <= 1e-2 * want + 1e-3, (r, dev0[r], want)
    # rows never kept at a layer hold the reused cache: stored V, re-rotated stored K
    for l in (0, L // 2, L - 1):
        kept = set(sels[l].tolist())
        for r in [int(x) for x in rng.choice(C, 24, replace=False) if int(x) not in kept][:8]:
            ci, j = divmod(r, req.chunk_len)
            st = store.chunks[ids[ci]]
            np.testing.assert_array_equal(f32(fr.V[l][r]), f32(st.V[l][j]))
            want = O.rope_reposition(f32(st.K[l][j:j + 1]), ci * req.chunk_len, spec.theta)[0]
            assert_close(f32(fr.K[l][r]), want, atol=1e-6, rtol=2.0 ** -8, what=f"reused K layer {l}")
