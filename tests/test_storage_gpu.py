"""Storage tier: chunk K/V read from files layer by layer while earlier layers recompute
(QCFuse technical summary, section 2.A: chunk KV on SSD, anchors in CPU memory, layer
i+1 loaded while layer i is recomputed).

A request served from files must give bit for bit what it gives from pinned host
memory (the same bytes reach the same kernels); a short file is reported by
qcf_storage_status without touching device memory outside the request.
"""
import os

import numpy as np
import pytest
import torch

import qcfdata as qd
from oracle import qcf_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def world():
    from rag_kv_cache_re_gb300 import model as M
    spec, req = qd.TINY, qd.TINY_REQ
    weights = qd.ModelWeights(spec)
    dm = M.DeviceModel(weights, DEV, max_pos=256)
    om = O.OracleModel(weights)
    store = M.ChunkStore(dm, req.crit_layer, req.n_anchor)
    for c in range(4):
        t = qd.chunk_tokens(c, req.chunk_len, spec.vocab)
        k = O.chunk_precompute(om, t)
        store.add_precomputed(c, t, torch.from_numpy(k["K"]).to(torch.bfloat16), torch.from_numpy(k["V"]).to(torch.bfloat16))
    return dict(M=M, spec=spec, req=req, dm=dm, store=store)


def _outputs(fr):
    return ([k.clone() for k in fr.K], [v.clone() for v in fr.V], fr.selected.clone(), fr.scores.clone(),
            fr.logits.clone(), fr.x_rows.clone())


@pytest.mark.parametrize("o_direct", [False, True], ids=["buffered", "o_direct"])
def test_storage_equals_pinned_host(world, tmp_path, o_direct):
    from rag_kv_cache_re_gb300 import qcf as Q
    w = world
    M, req = w["M"], w["req"]
    ids = [2, 0, 3]
    q = qd.query_tokens(5, req.query_len, w["spec"].vocab)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    ref = M.FusedRequest(w["dm"], w["store"], ids, q, req.ratio_bp)
    ref.run(cs, xs)
    torch.cuda.synchronize()
    want = _outputs(ref)
    files = M.ChunkFiles(w["store"], str(tmp_path), o_direct=o_direct)
    nbytes = files.write(ids)
    assert nbytes == sum(w["store"].chunks[c].K.numel() * 2 * 2 for c in ids)
    fr = M.FusedRequest(w["dm"], w["store"], ids, q, req.ratio_bp)
    for _ in range(2):   # twice: the pinned double buffer is reused across requests
        fr.run_from_storage(files, cs, xs)
        torch.cuda.synchronize()
        assert Q.qcf_storage_status() == 0 and Q.qcf_query_status() == 0
        got = _outputs(fr)
        for a, b in zip(got[0] + got[1], want[0] + want[1]):
            assert torch.equal(a, b)
        for a, b in zip(got[2:], want[2:]):
            assert torch.equal(a, b)
    files.close()


def test_storage_short_file_is_reported(world, tmp_path):
    from rag_kv_cache_re_gb300 import qcf as Q
    w = world
    M, req = w["M"], w["req"]
    ids = [1, 2, 3]
    q = qd.query_tokens(6, req.query_len, w["spec"].vocab)
    files = M.ChunkFiles(w["store"], str(tmp_path), o_direct=False)
    files.write(ids)
    victim = files.paths[M.ChunkStore.content_key(w["store"].chunks[3].tokens)]
    size = os.path.getsize(victim)
    with open(victim, "r+b") as f:
        f.truncate(size // 2)   # the keys stay, the values of every layer are gone
    fr = M.FusedRequest(w["dm"], w["store"], ids, q, req.ratio_bp)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    fr.run_from_storage(files, cs, xs)
    torch.cuda.synchronize()
    assert Q.qcf_storage_status() != 0      # the short read, reported once
    assert Q.qcf_storage_status() == 0
    assert Q.qcf_query_status() == 0        # nothing on the device noticed: no fault
    files.close()
