"""Host-side logic the product and the bench rely on (CPU only): the seeded input
generators, the KV-deviation selector's layer schedule, the content-keyed chunk
store, and the guard that keeps recorded ncu traffic tied to the sources it
describes."""
import hashlib
import json
import os

import numpy as np
import pytest

import qcfdata as qd
import bench
from rag_kv_cache_re_gb300.model import ChunkStore, StoredChunk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("n,frac", [(10, 0.70), (35, 0.70), (8, 0.5), (5, 1.0), (6, 0.0)])
def test_shared_chunk_requests(n, frac):
    a, b = qd.shared_chunk_requests(n, frac)
    assert len(a) == n and len(b) == n
    assert len(set(a.tolist())) == n and len(set(b.tolist())) == n   # no repeats inside a request
    assert len(set(a.tolist()) & set(b.tolist())) == int(np.floor(frac * n + 0.5))
    a2, b2 = qd.shared_chunk_requests(n, frac)                        # seeded: the same lists again
    assert np.array_equal(a, a2) and np.array_equal(b, b2)


@pytest.mark.parametrize("pattern", ["uniform", "clusters"])
@pytest.mark.parametrize("C,N", [(100, 15), (4096, 410), (16, 16), (10, 0), (5120, 768)])
def test_selected_indices(pattern, C, N):
    idx = qd.selected_indices(C, N, pattern)
    assert idx.dtype == np.int32 and len(idx) == N
    if N:
        assert idx[0] >= 0 and idx[-1] < C
        assert np.all(np.diff(idx) > 0)                               # strictly ascending, distinct
    assert np.array_equal(idx, qd.selected_indices(C, N, pattern))
    if pattern == "clusters" and N:
        runs = 1 + int(np.sum(np.diff(idx) > 1))
        assert runs <= 8


def test_selected_indices_rejects_unknown_pattern():
    with pytest.raises(ValueError):
        qd.selected_indices(100, 10, "stripes")


@pytest.mark.parametrize("L,r", [(32, 1500), (32, 3000), (80, 5000), (2, 2500)])
def test_hkvd_schedule(L, r):
    s = bench.hkvd_schedule(L, r)
    assert len(s) == L and s[0] == 2 * r and s[-1] == r
    # what the library checks before a KV-deviation request runs
    assert all(0 <= v <= 10000 for v in s)
    assert all(x >= y for x, y in zip(s, s[1:]))


def _chunk(tokens):
    return StoredChunk(np.asarray(tokens, np.int32), None, None, np.zeros(0, np.int32), None, None)


def test_chunk_store_keys_chunks_by_content():
    store = ChunkStore(model=None, crit_layer=1, n_anchor=0)
    t = np.arange(40, dtype=np.int64) * 7 % 101
    assert ChunkStore.content_key(t) == ChunkStore.content_key(t.astype(np.int32))
    assert ChunkStore.content_key(t) != ChunkStore.content_key(t[::-1].copy())
    c = store._keep(3, _chunk(t))
    # another id with the same tokens maps to the stored chunk; different tokens do not
    assert store._known(9, t.astype(np.int32)) is c and store.chunks[9] is c
    assert store._known(10, t + 1) is None and 10 not in store.chunks


def test_recorded_traffic_follows_the_sources():
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    rec = json.load(open(path))["gemm_gate_up_swiglu"]
    h = hashlib.sha256()
    for f in rec["sources"]:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    got = bench.recorded_traffic("gemm_gate_up_swiglu")
    if h.hexdigest() == rec["sources_sha256"]:
        assert got == rec["traffic_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    else:
        assert got is None
    assert bench.recorded_traffic("no_such_kernel") is None


def test_per_device_setup_runs_once_for_each_device(tmp_path):
    """Kernel attributes (the dynamic shared-memory limit) and symbol addresses belong to
    one device: the library's set-up helper must run once per device, keep each device's
    result apart, and survive concurrent first calls.  Compiled from the library's own
    header with the host compiler and driven with fake device indices (no GPU)."""
    import shutil
    import subprocess
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    hdr = os.path.join(ROOT, "rag_kv_cache_re_gb300", "csrc")
    src = tmp_path / "per_device_test.cpp"
    src.write_text(r'''
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <thread>
#include <vector>
#include "per_device.h"
int main() {
  qcf::PerDevice<int> pd;
  std::atomic<int> calls[4] = {};
  std::vector<std::thread> th;
  for (int t = 0; t < 16; ++t)
    th.emplace_back([&, t] {
      const int dev = t % 3;
      for (int k = 0; k < 100; ++k) {
        const int v = pd.get(dev, [&] { calls[dev]++; return 100 + dev; });
        if (v != 100 + dev) { std::printf("wrong value %d on device %d\n", v, dev); std::_Exit(2); }
      }
    });
  for (auto& x : th) x.join();
  for (int d = 0; d < 3; ++d)
    if (calls[d] != 1) { std::printf("device %d set up %d times\n", d, calls[d].load()); return 3; }
  int uncached = 0;   // an unreadable device (-1) is never cached
  pd.get(-1, [&] { return ++uncached; });
  pd.get(-1, [&] { return ++uncached; });
  if (uncached != 2) return 4;
  // device 7 first: the table grows, earlier devices keep their values
  if (pd.get(7, [] { return 7; }) != 7 || pd.get(1, [] { return -1; }) != 101) return 5;
  std::puts("ok");
  return 0;
}
''')
    exe = tmp_path / "per_device_test"
    subprocess.run([gxx, "-std=c++17", "-O1", "-pthread", "-I", hdr, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_chunk_files_layout(tmp_path):
    """ChunkFiles writes a chunk as raw bf16 keys [L][len][Hkv][D] then values, named by
    content, once per content; the offsets it hands the library address those blocks."""
    import torch
    from rag_kv_cache_re_gb300.model import ChunkFiles
    L, n, Hkv, D = 3, 8, 2, 16
    g = torch.Generator().manual_seed(0)

    def chunk(seed):
        K = torch.randn((L, n, Hkv, D), generator=g).to(torch.bfloat16)
        V = torch.randn((L, n, Hkv, D), generator=g).to(torch.bfloat16)
        return StoredChunk(np.arange(n, dtype=np.int32) + seed, K, V, np.zeros(0, np.int32), None, None)

    class _Store:
        chunks = {0: chunk(0), 1: chunk(100)}

    _Store.chunks[2] = _Store.chunks[0]            # same content: one file
    files = ChunkFiles(_Store, str(tmp_path), o_direct=False)
    assert files.write([0, 1, 2]) == 2 * 2 * L * n * Hkv * D * 2
    assert len(os.listdir(tmp_path)) == 2
    c = _Store.chunks[1]
    raw = open(files.paths[ChunkStore.content_key(c.tokens)], "rb").read()
    block = n * Hkv * D * 2
    for l in range(L):
        k = np.frombuffer(raw[l * block:(l + 1) * block], dtype=np.int16)
        v = np.frombuffer(raw[(L + l) * block:(L + l + 1) * block], dtype=np.int16)
        assert np.array_equal(k, c.K[l].contiguous().view(torch.int16).numpy().ravel())
        assert np.array_equal(v, c.V[l].contiguous().view(torch.int16).numpy().ravel())
