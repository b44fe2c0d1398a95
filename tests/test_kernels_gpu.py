"""Parity of every qcf_* kernel entry point with the CPU oracle (GPU).

Inputs come from qcdata's seeded generators; expected values from oracle/ only.
Sizes span several tiles with ragged tails; full-size sweep points are checked
through properties that hold at any size.
"""
import math

import numpy as np
import pytest
import torch

import qcfdata as qd
from oracle import qcf_oracle as O
from _parity import assert_close, assert_same_selection

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Q():
    from rag_kv_cache_re_gb300 import qcf
    return qcf


DEV = "cuda"


def f32(t):
    return t.float().cpu().numpy()


def table(Q, max_pos, D):
    return Q.RopeTable(max_pos, D, 1e4, DEV)


# ----------------------------------------------------------------- RoPE re-rotation

@pytest.mark.parametrize("D,Hkv", [(16, 4), (128, 8)])
@pytest.mark.parametrize("inplace", [False, True])
def test_rope_reposition(Q, D, Hkv, inplace):
    lens = [37, 512, 3, 200]
    start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    delta = np.array([0, 5000, 131000, 77], np.int32)
    K = qd.normal_bf16((int(start[-1]), Hkv, D), 1.0, 11, DEV)
    src = K.clone()
    dst = K if inplace else torch.empty_like(K)
    Q.qcf_rope_reposition(K, dst, start, delta, table(Q, 131200, D))
    torch.cuda.synchronize()
    ref = np.concatenate([O.rope_reposition(f32(src[start[s]:start[s + 1]]), delta[s], 1e4) for s in range(len(lens))])
    got = f32(dst)
    # bf16 output: within one rounding of the exact rotation (fp32 table)
    assert_close(got, ref, atol=1e-6, rtol=2.0 ** -8, what="reposition")
    assert_close(got, ref, atol=2e-2, rtol=2e-2, what="reposition (stated tolerance)")


# ----------------------------------------------------------------- anchors

@pytest.mark.parametrize("D,Hkv,lens,A", [(16, 4, [32, 32, 32], 2), (128, 8, [512] * 10, 8), (128, 8, [700, 9, 1024], 8)])
def test_anchor_keynorm_topk(Q, D, Hkv, lens, A):
    start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    K = qd.normal_bf16((int(start[-1]), Hkv, D), 1.0, 12, DEV)
    K[5] = K[1]                      # exact norm tie inside chunk 0: lower index wins
    idx, norms = Q.qcf_anchor_keynorm_topk(K, start, A, want_norms=True)
    torch.cuda.synchronize()
    Kh = f32(K)
    ref_idx = O.keynorm_anchors(Kh, start, A)
    got = idx.cpu().numpy()
    for c in range(len(lens)):
        rows = Kh[start[c]:start[c + 1]].astype(np.float64)
        nrm = np.sqrt(np.sum(rows.reshape(rows.shape[0], -1) ** 2, axis=1))
        assert np.all(np.diff(got[c]) > 0), "anchors must be ascending"
        assert_same_selection(got[c], nrm, A, tie_tol=1e-5 * nrm.max(), what=f"anchors chunk {c}")
    assert (5 not in got[0]) or (1 in got[0]), "equal norms: the lower index must be taken first"
    assert ref_idx.shape == got.shape
    ref_n = np.sqrt(np.sum(Kh.astype(np.float64).reshape(Kh.shape[0], -1) ** 2, axis=1))
    assert_close(norms.cpu().numpy(), ref_n, atol=1e-4, rtol=1e-5, what="norms")


# ----------------------------------------------------------------- profiling

@pytest.mark.parametrize("C,nq,Hq,Hkv,D,scale", [
    (96, 8, 4, 4, 16, 0.25),       # tiny model shape
    (300, 64, 32, 8, 128, 1.0),    # ragged tail, sweep distributions
    (4096, 64, 32, 8, 128, 1.0),   # sweep 4k
    (5120, 64, 32, 8, 128, 1.0 / math.sqrt(128)),  # 8B request shape
    (16384, 64, 32, 8, 128, 1.0),  # sweep 16k
    (2000, 128, 56, 8, 128, 1.0),  # 34B head layout (7 heads per KV head, 4 row groups)
    (3000, 64, 64, 8, 128, 1.0),   # 70B head layout (8 heads per KV head, 2 row groups)
    (129, 50, 32, 8, 128, 1.0),    # ragged keys, a partial row tile
    (1, 64, 32, 8, 128, 1.0),      # a single key
    (777, 100, 8, 8, 128, 1.0),    # no grouping: one row tile of 100 rows
    (1500, 20, 128, 8, 128, 1.0),  # 16 heads per KV head: 3 row tiles, the second group has one
    (4096, 64, 32, 8, 128, 8.0),   # a sharp softmax (a few keys carry each row)
])
def test_profile_scores(Q, C, nq, Hq, Hkv, D, scale):
    t = qd.sweep_tensors(C, n_query=nq, Hq=Hq, Hkv=Hkv, D=D, device=DEV)
    s = Q.qcf_profile_scores(t["Q"], t["K"], scale)
    torch.cuda.synchronize()
    ref = O.profile_scores(f32(t["Q"]), f32(t["K"]), scale)
    assert_close(s.cpu().numpy(), ref, atol=1e-3, rtol=1e-3, what="scores")
    assert abs(float(s.double().sum()) - Hq * nq) < 1e-3 * Hq * nq


@pytest.mark.parametrize("C", [65536, 131072])
def test_profile_scores_full_size_properties(Q, C):
    t = qd.sweep_tensors(C, device=DEV)
    s = Q.qcf_profile_scores(t["Q"], t["K"], 1.0)
    torch.cuda.synchronize()
    v = s.double().cpu().numpy()
    assert np.all(v >= 0) and np.all(np.isfinite(v))
    assert abs(v.sum() - 32 * 64) < 1e-3 * 32 * 64
    # the keys with equal K get equal scores: plant a duplicate key and compare
    K2 = t["K"].clone()
    K2[C - 1] = K2[7]
    s2 = Q.qcf_profile_scores(t["Q"], K2, 1.0).cpu().numpy()
    assert abs(s2[C - 1] - s2[7]) <= 1e-6 * max(1e-30, abs(s2[7])) + 1e-9


# ----------------------------------------------------------------- top-N

@pytest.mark.parametrize("C", [1, 7, 1000, 5120, 16384, 16385, 20480, 131072, 1 << 20])
def test_topn_select_exact(Q, C):
    # 16384 scores or fewer are resolved in shared memory alone; above that a histogram
    # pass narrows them to one bucket first; one value repeated 20000+ times overflows the
    # bucket list and takes the all-global radix path
    rng = np.random.default_rng(C)
    for kind in ("ties", "continuous", "negative", "one_value"):
        if kind == "ties":
            v = (rng.integers(0, 9, C) * 0.125).astype(np.float32)
            v[rng.integers(0, C, max(1, C // 10))] = -0.0
        elif kind == "negative":
            v = (rng.standard_normal(C) * 1e3).astype(np.float32)
        elif kind == "one_value":
            v = np.full(C, 0.375, np.float32)
            v[rng.integers(0, C, max(1, C // 100))] = 1.5
        else:
            v = rng.random(C, dtype=np.float32) * 2.0
        s = torch.from_numpy(v).to(DEV)
        for N in sorted({0, 1, max(0, C // 7), O.num_selected(C, 1500), C - 1, C}):
            if N < 0:
                continue
            got = Q.qcf_topn_select(s, N).cpu().numpy()
            want = O.topn_select(v.astype(np.float64), N)
            assert np.array_equal(got, want), f"C={C} N={N} {kind}"


@pytest.mark.parametrize("C", [100, 16385, 20480, 131072, 300001, 152 * 4096, 1 << 20])
def test_topn_select_grid_exact(Q, C):
    # above 16384 scores the workspace entry point spreads over a cooperative grid (4096
    # scores per CTA); uniform [1, 2) shares its top 11 key bits, so it needs a second
    # global level; one value repeated fixes every key bit and ranks the equal keys by
    # index across CTAs; beyond one resident grid the call is the one-CTA kernel
    rng = np.random.default_rng(C + 1)
    ws = Q.workspace(Q._lib.lib().qcf_topn_select_workspace_size(C), DEV, "topn_test")
    ws.fill_(0xFF)   # the scratch needs no clearing: every call resets what it uses
    for kind in ("ties", "continuous", "unit_interval", "one_value", "negative"):
        if kind == "ties":
            v = (rng.integers(0, 9, C) * 0.125).astype(np.float32)
            v[rng.integers(0, C, max(1, C // 10))] = -0.0
        elif kind == "unit_interval":
            v = (1.0 + rng.random(C, dtype=np.float32)).astype(np.float32)
        elif kind == "one_value":
            v = np.full(C, 0.375, np.float32)
            v[rng.integers(0, C, max(1, C // 100))] = 1.5
        elif kind == "negative":
            v = (rng.standard_normal(C) * 1e3).astype(np.float32)
        else:
            v = rng.random(C, dtype=np.float32) * 2.0
        s = torch.from_numpy(v).to(DEV)
        for N in sorted({1, 7, O.num_selected(C, 1500), C // 2 + 3, C}):
            got = Q.qcf_topn_select_ws(s, N, ws).cpu().numpy()
            want = O.topn_select(v.astype(np.float64), N)
            assert np.array_equal(got, want), f"C={C} N={N} {kind}"
    assert Q.qcf_query_status() == 0


# ----------------------------------------------------------------- gather / scatter

def test_gather_and_scatter_exact(Q):
    src = qd.normal_bf16((1000, 8, 128), 1.0, 13, DEV)
    idx = torch.tensor(qd.selected_indices(1000, 77, "uniform"), dtype=torch.int32, device=DEV)
    g = Q.qcf_gather_rows(src, idx)
    assert torch.equal(g, src[idx.long()])
    Kc = qd.normal_bf16((1000, 8, 128), 1.0, 14, DEV)
    Vc = qd.normal_bf16((1000, 8, 128), 1.0, 15, DEV)
    K0, V0 = Kc.clone(), Vc.clone()
    kn = qd.normal_bf16((77, 8, 128), 1.0, 16, DEV)
    vn = qd.normal_bf16((77, 8, 128), 1.0, 17, DEV)
    Q.qcf_scatter_kv(kn, vn, idx, Kc, Vc)
    K0[idx.long()] = kn
    V0[idx.long()] = vn
    assert torch.equal(Kc, K0) and torch.equal(Vc, V0)
    assert Q.qcf_query_status() == 0


def test_bad_index_sets_status_without_fault(Q):
    src = qd.normal_bf16((10, 8), 1.0, 18, DEV)
    idx = torch.tensor([1, 10, 3], dtype=torch.int32, device=DEV)   # 10 is out of range
    Q.qcf_gather_rows(src, idx)
    assert Q.qcf_query_status() & 0x2
    assert Q.qcf_query_status() == 0                                  # read clears


# ----------------------------------------------------------------- sparse causal attention

@pytest.mark.parametrize("T,n,Hq,Hkv,D,pattern", [
    (104, 23, 4, 4, 16, "uniform"),        # tiny fused shape (15 selected + 8 query)
    (104, 104, 4, 4, 16, "all"),           # tiny full prefill (dense causal)
    (300, 1, 32, 8, 128, "first"),         # a single row at position 0
    (1000, 150, 32, 8, 128, "clusters"),
    (5184, 832, 32, 8, 128, "uniform"),    # 8B request shape: 768 selected + 64 query
    (2000, 300, 56, 8, 128, "uniform"),    # 34B head layout (G = 7)
])
def test_sparse_causal_attn(Q, T, n, Hq, Hkv, D, pattern):
    if pattern == "all":
        pos = np.arange(T)
    elif pattern == "first":
        pos = np.array([0])
    else:
        Cx = T - 64 if T > 600 else T - 8
        nsel = n - (T - Cx)
        pos = np.concatenate([qd.selected_indices(Cx, nsel, pattern), np.arange(Cx, T)])
    pos = pos.astype(np.int32)
    assert len(pos) == n
    K = qd.normal_bf16((T, Hkv, D), 1.0, 21, DEV)
    V = qd.normal_bf16((T, Hkv, D), 1.0, 22, DEV)
    q = qd.normal_bf16((n, Hq, D), 1.0, 23, DEV)
    scale = 1.0 / math.sqrt(D)
    o, lse = Q.qcf_sparse_causal_attn(q, torch.from_numpy(pos).to(DEV), K, V, scale, want_lse=True)
    torch.cuda.synchronize()
    ref = O.causal_attention(f32(q), pos, f32(K), f32(V), scale)
    assert_close(f32(o), ref, atol=2e-2, rtol=2e-2, what="attention output")
    # lse: natural log of sum_j exp(scale q.k_j) over visible keys
    qd64, Kd = f32(q).astype(np.float64), f32(K).astype(np.float64)
    G = Hq // Hkv
    for r in list(range(0, n, max(1, n // 5)))[:5]:
        for h in (0, Hq - 1):
            s = scale * Kd[: pos[r] + 1, h // G] @ qd64[r, h]
            want = s.max() + np.log(np.exp(s - s.max()).sum())
            assert abs(float(lse[r, h]) - want) < 1e-3 * max(1.0, abs(want))
    assert Q.qcf_query_status() == 0


@pytest.mark.parametrize("T,n,Hq,Hkv,D", [(5184, 832, 32, 8, 128), (300, 45, 4, 4, 64), (96, 23, 4, 4, 16)])
def test_sparse_causal_attn_writes_only_its_rows(Q, T, n, Hq, Hkv, D):
    # the C ABI writes o [n][Hq][D]: rows after n in the caller's buffer stay as they were,
    # and the result equals the binding's own allocation bit for bit
    Cx = T - 64 if T > 600 else T - 8
    pos = np.concatenate([qd.selected_indices(Cx, n - (T - Cx), "uniform"), np.arange(Cx, T)]).astype(np.int32)
    K = qd.normal_bf16((T, Hkv, D), 1.0, 24, DEV)
    V = qd.normal_bf16((T, Hkv, D), 1.0, 25, DEV)
    q = qd.normal_bf16((n, Hq, D), 1.0, 26, DEV)
    p = torch.from_numpy(pos).to(DEV)
    o = Q.qcf_sparse_causal_attn(q, p, K, V, 1.0 / math.sqrt(D))
    o_g = torch.full((n + 16, Hq, D), 3.0, device=DEV, dtype=torch.bfloat16)
    ws = Q.workspace(Q._lib.lib().qcf_sparse_causal_attn_workspace_size(n, T, Hq, Hkv, D), q.device)
    Q.call("qcf_sparse_causal_attn", Q._ptr(q), Q._ptr(p), n, Q._ptr(K), Q._ptr(V), T, Hq, Hkv, D,
           float(1.0 / math.sqrt(D)), Q._ptr(o_g), None, Q._ptr(ws), ws.numel(), Q._stream(None))
    torch.cuda.synchronize()
    assert torch.equal(o_g[:n], o)
    assert bool((o_g[n:] == 3.0).all()), "attention wrote past row n"


# ----------------------------------------------------------------- dense pieces

@pytest.mark.parametrize("M,N,K", [(23, 192, 64), (1, 64, 64), (300, 384, 192), (832, 6144, 4096), (832, 4096, 4096), (832, 28672, 4096),
                                   (64, 4096, 14336), (832, 4096, 14336), (200, 28672, 256),
                                   # two 128-row tiles, the second ragged
                                   (129, 6144, 4096), (144, 28672, 4096), (144, 4096, 4096), (256, 4096, 14336),
                                   # the 8B layer shapes at the recompute and probe row counts: grouped stream-K
                                   # with staged fixups in one or two column passes, the lockstep staged
                                   # residual add, k splits with staged partials
                                   (832, 6144, 4096), (832, 28672, 4096), (832, 4096, 4096), (832, 4096, 14336),
                                   (1664, 4096, 14336), (64, 6144, 4096), (64, 4096, 14336),
                                   # tiles ending inside a warp's 32 rows (staged copies and stores past M)
                                   (837, 4096, 14336), (837, 6144, 4096), (100, 4096, 14336),
                                   # residual adds on 224-wide tiles with a ragged last column tile of 64
                                   # or 32 columns (and a row tail): no column past N may be written
                                   (256, 512, 128), (300, 256, 64), (837, 4096, 4096)])
def test_linear_store_and_add(Q, M, N, K):
    A = qd.normal_bf16((M, K), 1.0, 31, DEV)
    W = qd.normal_bf16((N, K), 0.02, 32, DEV)
    ref = (f32(A) @ f32(W).T).astype(np.float64)   # fp32 BLAS: error far below the tolerances used
    # outputs are the first M rows of buffers with 64 guard rows after them, which
    # no epilogue path (direct, staged, TMA-stored) may touch
    out_g = torch.full((M + 64, N), 7.0, device=DEV, dtype=torch.bfloat16)
    Q.qcf_linear(A, W, out=out_g[:M])
    torch.cuda.synchronize()
    assert_close(f32(out_g[:M]), ref, atol=1e-3, rtol=2.0 ** -8, what="bf16 out")
    assert bool((out_g[M:] == 7.0).all()), "bf16 store wrote past row M"
    base_g = torch.randn((M + 64, N), device=DEV, dtype=torch.float32)
    b0 = base_g.cpu().numpy().astype(np.float64)
    Q.qcf_linear(A, W, out=base_g[:M], add=True)
    torch.cuda.synchronize()
    # fp32 accumulation: each of the K/16 tensor-core steps may round the running
    # sum once (2^-23 relative); bound by the result's scale
    acc_tol = (K / 16) * 2.0 ** -22 * max(1.0, float(np.sqrt(np.mean(ref ** 2))))
    got = base_g.cpu().numpy()
    assert_close(got[:M], b0[:M] + ref, atol=max(1e-5, acc_tol), rtol=1e-5, what="fp32 residual add")
    assert np.array_equal(got[M:], b0[M:].astype(np.float32)), "residual add wrote past row M"


@pytest.mark.parametrize("M,N,K", [(832, 4096, 14336), (64, 4096, 14336), (832, 6144, 4096), (837, 4096, 14336)])
def test_linear_shared_tiles_deterministic(Q, M, N, K):
    # shared tiles are summed in slot order whichever unit arrives last: repeated
    # launches give the same bits
    A = qd.normal_bf16((M, K), 1.0, 36, DEV)
    W = qd.normal_bf16((N, K), 0.02, 37, DEV)
    first = Q.qcf_linear(A, W)
    x0 = torch.randn((M, N), device=DEV, dtype=torch.float32)
    x1 = x0.clone()
    Q.qcf_linear(A, W, out=x0, add=True)
    for _ in range(3):
        assert torch.equal(Q.qcf_linear(A, W), first)
    Q.qcf_linear(A, W, out=x1, add=True)
    torch.cuda.synchronize()
    assert torch.equal(x0, x1)


@pytest.mark.parametrize("M,N,K", [(23, 64, 64), (300, 384, 192), (832, 4096, 4096), (64, 4096, 14336)])
def test_linear_weights_stored_k_by_n(Q, M, N, K):
    # W kept [K][N] (N contiguous): the tensor cores read it as an MN-major operand
    A = qd.normal_bf16((M, K), 1.0, 34, DEV)
    Wkn = qd.normal_bf16((K, N), 0.02, 35, DEV)
    ref = (f32(A) @ f32(Wkn)).astype(np.float64)
    out = Q.qcf_linear(A, Wkn, w_kn=True)
    torch.cuda.synchronize()
    assert_close(f32(out), ref, atol=1e-3, rtol=2.0 ** -8, what="bf16 out, W [K][N]")
    base = torch.zeros((M, N), device=DEV, dtype=torch.float32)
    Q.qcf_linear(A, Wkn, out=base, add=True, w_kn=True)
    torch.cuda.synchronize()
    acc_tol = (K / 16) * 2.0 ** -22 * max(1.0, float(np.sqrt(np.mean(ref ** 2))))
    assert_close(base.cpu().numpy(), ref, atol=max(1e-5, acc_tol), rtol=1e-5, what="fp32 add, W [K][N]")


def test_rmsnorm(Q):
    x = torch.randn((300, 4096), device=DEV) * 3
    g = qd.normal_bf16((4096,), 1.0, 33, DEV)
    h = Q.qcf_rmsnorm(x, g, 1e-5)
    ref = O.rmsnorm(x.cpu().numpy(), f32(g), 1e-5)
    assert_close(f32(h), ref, atol=1e-6, rtol=2.0 ** -8, what="rmsnorm")
