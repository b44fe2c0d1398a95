"""Benchmark: fused RAG prefill (query-centric KV-cache fusion) vs full prefill on one GB300.

Workload: a Llama-3-8B-shaped random-init bf16 decoder (32 layers, d 4096, 32 Q /
8 KV heads, head dim 128, FFN 14336, vocab 128256, weights N(0, 0.02)); one
request of 10 retrieved chunks x 512 tokens + 64 query tokens (uniform ids),
critical layer 16, 15 % recompute (N = 768), 8 anchors per chunk.  The chunks'
per-layer K/V are precomputed offline on the GPU, each chunk alone, and kept in
pinned host memory; every step streams them back layer by layer as the method
prescribes.

A step is one fused prefill: probe, critical-layer profiling, top-N, 32 layers
of selective recompute with the next layers' K/V copied on a side stream, LM
head, first token on the host.  value = context tokens per second = C / step
time.  e2e repeats the step through the same public API with the token ids
copied from pinned host memory and the logits and first token copied back.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With N > 1 (torchrun) every rank runs an independent replica on its own GPU
(the path has no exchange step); value = all ranks' context tokens / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import qcfdata as qd  # noqa: E402

METRIC = "fused-prefill context tokens/s + TTFT ms at 15% recompute vs full prefill"
UNIT = "context tokens/s"
WORKLOAD = ("llama3-8b-shaped fused RAG prefill: 10 chunks x 512 + 64 query tokens, critical layer 16, "
            "15% recompute (N=768), 8 anchors/chunk, chunk K/V streamed from pinned host")


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of `value` over the ranks of the default process group (identity at world 1)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu record, only if the kernel's
    sources are unchanged since the counters were taken (else None)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec:
        return None
    h = hashlib.sha256()
    for f in rec["sources"]:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return rec["traffic_bytes_per_launch"] if h.hexdigest() == rec["sources_sha256"] else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d.get("hbm_gbs", 6791.0), "bf16": d.get("bf16_tflops", 1900.8),
                "bf16_sustained": d.get("bf16_tflops_sustained", 1702.3), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------- the workload

def build_workload(device, spec=qd.LLAMA8B, req=qd.LLAMA8B_REQ):
    from rag_kv_cache_re_gb300 import model as M
    weights = qd.ModelWeights(spec, device=str(device))
    dm = M.DeviceModel(weights, device, max_pos=8192)
    del weights
    torch.cuda.empty_cache()
    store = M.ChunkStore(dm, req.crit_layer, req.n_anchor)
    chunk_ids = list(range(req.n_chunks))
    for c in chunk_ids:   # offline: each chunk prefilled alone at positions 0..511
        store.ingest(c, qd.chunk_tokens(c, req.chunk_len, spec.vocab))
    query = qd.query_tokens(0, req.query_len, spec.vocab)
    fr = M.FusedRequest(dm, store, chunk_ids, query, req.ratio_bp)
    return dm, store, fr


def gemm_flops(spec, n_rows, ffn_padded):
    d, D = spec.d_model, spec.head_dim
    return {"gemm_qkv_rope": 2.0 * n_rows * d * (spec.n_heads + 2 * spec.n_kv_heads) * D,
            "gemm_o_resid": 2.0 * n_rows * spec.n_heads * D * d,
            "gemm_gate_up_swiglu": 2.0 * n_rows * d * 2 * ffn_padded,
            "gemm_down_resid": 2.0 * n_rows * ffn_padded * d}


def hkvd_schedule(L, ratio_bp):
    """Kept share per layer for the KV-deviation selector: 2r at layer 0 falling linearly to r."""
    sched = [int(round(2 * ratio_bp - ratio_bp * l / (L - 1))) for l in range(L)]
    sched[-1] = ratio_bp
    return sched


def time_selectors(dm, store, fr, spec, req, cs, xs, reps):
    """TTFT (CUDA events on the compute stream) of the selector variants on the same chunks and query."""
    from rag_kv_cache_re_gb300 import model as M
    store_last = M.ChunkStore(dm, spec.n_layers - 1, req.n_anchor)   # QCLast: anchors and profile at the last layer
    for c in fr.chunk_ids:
        store_last.ingest(c, store.chunks[c].tokens)
    query = fr.ids_host[fr.C:].numpy()
    sched = hkvd_schedule(spec.n_layers, req.ratio_bp)
    variants = {
        "qclast": M.FusedRequest(dm, store_last, fr.chunk_ids, query, req.ratio_bp),
        "qcall": M.FusedRequest(dm, store, fr.chunk_ids, query, req.ratio_bp, selector=M.SELECT_ALL_LAYERS),
        "hkvd": M.FusedRequest(dm, store, fr.chunk_ids, query, req.ratio_bp, selector=M.SELECT_HKVD,
                               layer_ratio_bp=sched),
    }
    out = {}
    for name, v in variants.items():
        for _ in range(2):
            v.run(cs, xs)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cs)
        for _ in range(reps):
            v.run(cs, xs)
        e1.record(cs)
        torch.cuda.synchronize()
        out[f"{name}_ttft_ms"] = round(e0.elapsed_time(e1) / reps, 3)
    out["hkvd_schedule_bp"] = f"{sched[0]} at layer 0 falling linearly to {sched[-1]} at layer {spec.n_layers - 1}"
    out["hkvd_rows_per_layer"] = [n + fr.Q for n in variants["hkvd"].layer_N]
    del variants, store_last
    torch.cuda.empty_cache()
    return out


def time_dedupe(dm, store, fr, spec, req, cs, xs, reps):
    """Two 8B requests sharing 70 % of their chunks: one after the other vs one batch
    whose shared chunks cross the host link once per layer (TTFT of both, bytes sent)."""
    from rag_kv_cache_re_gb300 import model as M
    sets = qd.shared_chunk_requests(req.n_chunks, 0.70)
    for c in sorted(set(np.concatenate(sets).tolist())):
        if int(c) not in store.chunks:
            store.ingest(int(c), qd.chunk_tokens(int(c), req.chunk_len, spec.vocab))
    make = lambda: [M.FusedRequest(dm, store, list(map(int, ids)), qd.query_tokens(i, req.query_len, spec.vocab),
                                   req.ratio_bp) for i, ids in enumerate(sets)]
    seq, bat = make(), make()

    def run_seq():
        for r in seq:
            r.run(cs, xs)

    h2d = {}

    def run_bat():
        h2d["batch"] = M.run_batch(bat, cs, xs)

    out = {}
    for name, fn in (("sequential", run_seq), ("batched", run_bat)):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cs)
        for _ in range(reps):
            fn()
        e1.record(cs)
        torch.cuda.synchronize()
        out[f"{name}_ms"] = round(e0.elapsed_time(e1) / reps, 3)
    same = all(torch.equal(a.logits, b.logits) and torch.equal(a.selected, b.selected) for a, b in zip(seq, bat))
    per_req = sum(store.chunks[int(c)].K.numel() * 2 + store.chunks[int(c)].V.numel() * 2 for c in sets[0])
    anchors = sum(store.chunks[int(c)].aK[: req.crit_layer].numel() * 4 for ids in sets for c in ids)
    out.update({"requests": len(sets), "chunks_per_request": req.n_chunks,
                "distinct_chunks": len(set(np.concatenate(sets).tolist())),
                "h2d_bytes_sequential": int(2 * per_req + anchors), "h2d_bytes_batched": int(h2d["batch"]),
                "results_equal": bool(same)})
    del seq, bat
    torch.cuda.empty_cache()
    return out


def measure_host_link(fr, device):
    """Host link as the request uses it: one 256 MB pinned copy each way (the link's rate),
    and the request's own chunk-K/V copy pattern alone on a stream (one copy per chunk,
    layer and K or V: the copy engine's rate at these sizes)."""
    st = torch.cuda.Stream(device)
    big_h = torch.empty(256 << 20, dtype=torch.uint8).pin_memory()
    big_d = torch.empty(256 << 20, dtype=torch.uint8, device=device)

    def best_ms(fn, reps=3):
        best = 1e30
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(st)
            with torch.cuda.stream(st):
                fn()
            b.record(st)
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return best

    h2d_ms = best_ms(lambda: big_d.copy_(big_h, non_blocking=True))
    d2h_ms = best_ms(lambda: big_h.copy_(big_d, non_blocking=True))
    del big_h, big_d
    dst_k = [torch.empty_like(c.K[0], device=device) for c in fr.chunks]
    dst_v = [torch.empty_like(c.V[0], device=device) for c in fr.chunks]
    L = fr.chunks[0].K.shape[0]

    def pattern():
        for l in range(L):
            for c, dk, dv in zip(fr.chunks, dst_k, dst_v):
                dk.copy_(c.K[l], non_blocking=True)
                dv.copy_(c.V[l], non_blocking=True)

    pat_ms = best_ms(pattern)
    pat_bytes = sum(c.K.numel() * 2 + c.V.numel() * 2 for c in fr.chunks)
    n_copies = 2 * L * len(fr.chunks)
    return {"h2d_gb_per_s": round((256 << 20) / (h2d_ms * 1e-3) / 1e9, 1),
            "d2h_gb_per_s": round((256 << 20) / (d2h_ms * 1e-3) / 1e9, 1),
            "request_copies": {"copies": n_copies, "bytes": int(pat_bytes), "ms": round(pat_ms, 3),
                               "gb_per_s": round(pat_bytes / (pat_ms * 1e-3) / 1e9, 1)},
            "method": "256 MB pinned copies (best of 3); the request's chunk K/V copies alone on one stream"}


def time_storage_tier(dm, store, fr, cs, xs, reps):
    """TTFT of the same request with the chunks' K/V read from files layer by layer (the
    storage tier) instead of pinned host memory: O_DIRECT reads where the file system
    takes them (the device's own bandwidth), else buffered reads (page cache)."""
    from rag_kv_cache_re_gb300 import model as M
    from rag_kv_cache_re_gb300 import qcf as Q
    d = tempfile.mkdtemp(prefix="qcf_chunks_")
    out = {}
    try:
        for mode in ("o_direct", "buffered"):
            files = M.ChunkFiles(store, d, o_direct=mode == "o_direct")
            written = files.write(fr.chunk_ids)
            files.files_for(fr)
            if mode == "o_direct" and not files.o_direct:
                out["o_direct"] = {"unavailable": "the file system refused O_DIRECT"}
                files.close()
                continue
            fr.run_from_storage(files, cs, xs)
            torch.cuda.synchronize()
            ts = []
            for _ in range(reps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                a.record(cs)
                fr.run_from_storage(files, cs, xs)
                b.record(cs)
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b))
            err = Q.qcf_storage_status()
            read = sum(c.K.numel() * 2 + c.V.numel() * 2 for c in fr.chunks)
            ms = statistics.median(ts)
            out[mode] = {"ttft_ms": round(ms, 3), "bytes_read": int(read), "read_gb_per_s": round(read / (ms * 1e-3) / 1e9, 2),
                         "read_error": err, "bytes_on_storage": int(written) if written else None}
            files.close()
    finally:
        import shutil
        shutil.rmtree(d, ignore_errors=True)
    return out


def run_gpu(args):
    from rag_kv_cache_re_gb300 import qcf as Q
    world, rank, local = _dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    spec, req = qd.LLAMA8B, qd.LLAMA8B_REQ
    dm, store, fr = build_workload(device)
    cs, xs = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def step(e2e=False):
        fr.run(cs, xs, ids_from_host=e2e)
        if e2e:
            with torch.cuda.stream(cs):
                logits_host.copy_(fr.logits, non_blocking=True)

    logits_host = torch.empty(spec.vocab, dtype=torch.float32).pin_memory()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = Q.qcf_query_status()
    if status:
        raise RuntimeError(f"device status {status:#x} after warm-up")

    # ---- timed region: K fused prefills back to back (the headline TTFT and value)
    clocks = ClockSampler(device.index)
    barrier(world, device)
    torch.cuda.synchronize()
    clocks.start()
    launches0 = Q.qcf_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(cs)
    torch.cuda.nvtx.range_push("qcf_timed")
    for _ in range(args.steps):
        step()
    torch.cuda.nvtx.range_pop()
    ev1.record(cs)
    torch.cuda.synchronize()
    launches = Q.qcf_launch_count() - launches0
    # ---- the same K steps again with CUDA events around every library launch
    # (on the launching stream): per-kernel time and the roofline of the dominant kernel
    Q.qcf_timing_enable(True)
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0.record(cs)
    for _ in range(args.steps):
        step()
    k1.record(cs)
    torch.cuda.synchronize()
    per_kernel = Q.qcf_timing_read()
    Q.qcf_timing_enable(False)
    clk = clocks.stop()
    barrier(world, device)
    elapsed_ms = reduce_max_over_ranks(ev0.elapsed_time(ev1), world, device)
    ms_per_step = elapsed_ms / args.steps
    ms_with_events = k0.elapsed_time(k1) / args.steps
    C = fr.C
    value = world * C * args.steps / (elapsed_ms / 1e3)

    # ---- e2e: ids from pinned host, logits + first token back to the host, per step
    torch.cuda.synchronize()
    barrier(world, device)
    e0 = time.perf_counter()
    for _ in range(args.steps):
        step(e2e=True)
        cs.synchronize()
    e_ms = reduce_max_over_ranks((time.perf_counter() - e0) * 1e3, world, device)
    kv_bytes = sum(c.K.numel() * 2 + c.V.numel() * 2 for c in fr.chunks)
    anchor_bytes = sum(c.aK[: req.crit_layer].numel() * 2 + c.aV[: req.crit_layer].numel() * 2 for c in fr.chunks)
    h2d = int(fr.ids_host.numel() * 4 + kv_bytes + anchor_bytes)
    d2h = int(spec.vocab * 4 + 4)

    # ---- TTFT per request: each request alone, synchronised before and after (device time
    # from its first launch to the first token copied to the host), median over the requests
    def one_request_ms(run):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(cs)
        run()
        b.record(cs)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    n_ttft = args.ttft_requests
    fused_ttfts = [one_request_ms(lambda: fr.run(cs, xs)) for _ in range(n_ttft)]
    ttft_ms = reduce_max_over_ranks(statistics.median(fused_ttfts), world, device)

    # ---- full prefill on the same tokens (the baseline the ratio compares with)
    K_layers = [torch.empty((fr.T, spec.n_kv_heads, spec.head_dim), dtype=torch.bfloat16, device=device)
                for _ in range(spec.n_layers)]
    V_layers = [torch.empty_like(K_layers[0]) for _ in range(spec.n_layers)]
    tok_host = torch.zeros(1, dtype=torch.int32).pin_memory()

    def full_request():
        with torch.cuda.stream(cs):
            _, _, _, tok = Q.qcf_full_prefill(dm, fr.ids, K_layers, V_layers, stream=cs)
            tok_host.copy_(tok, non_blocking=True)

    for _ in range(2):
        full_request()
    torch.cuda.synchronize()
    full_ttfts = [one_request_ms(full_request) for _ in range(n_ttft)]
    full_ms = reduce_max_over_ranks(statistics.median(full_ttfts), world, device)
    n_full = max(2, min(5, args.steps))
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(cs)
    for _ in range(n_full):
        full_request()
    f1.record(cs)
    torch.cuda.synchronize()
    full_b2b_ms = reduce_max_over_ranks(f0.elapsed_time(f1) / n_full, world, device)

    # ---- the selector variants on the same request: QCLast, QCAll, CacheBlend HKVD
    selectors = None if args.no_selectors else time_selectors(dm, store, fr, spec, req, cs, xs, max(2, min(5, args.steps)))
    dedupe = None if args.no_selectors else time_dedupe(dm, store, fr, spec, req, cs, xs, max(2, min(5, args.steps)))
    storage = None if args.no_storage else time_storage_tier(dm, store, fr, cs, xs, 5)

    # ---- roofline of the dominant kernel (gate/up GEMM with SwiGLU epilogue)
    peaks = load_peaks()
    flops = gemm_flops(spec, fr.ns, dm.ffn_padded)
    total_ms = max(1e-9, sum(v[0] for v in per_kernel.values()))
    kernels = {name: {"ms_total": round(ms, 4), "launches": cnt, "share": round(ms / total_ms, 4)}
               for name, (ms, cnt) in per_kernel.items() if cnt > 0}
    # flops per step per GEMM class: 32 recompute layers of 832 rows (the probe's
    # 64-row GEMMs are timed apart, as probe_gemm)
    step_flops = {k: spec.n_layers * f for k, f in flops.items()}
    probe = gemm_flops(spec, req.query_len, dm.ffn_padded)
    step_flops["probe_gemm"] = sum(req.crit_layer * f for f in probe.values()) + \
        2.0 * req.query_len * spec.d_model * spec.n_heads * spec.head_dim
    for k, f in step_flops.items():
        if k in kernels:
            ms = kernels[k]["ms_total"] / args.steps
            kernels[k]["tflops"] = round(f / (ms * 1e-3) / 1e12, 1)
    if "probe_gemm" in kernels:   # weight-bound: report the weight bytes streamed per second
        wbytes = req.crit_layer * sum(t.numel() * 2 for k, t in dm.layer_tensors[0].items() if k.startswith("w_"))
        kernels["probe_gemm"]["weights_tb_per_s"] = round(wbytes / (kernels["probe_gemm"]["ms_total"] / args.steps * 1e-3) / 1e12, 2)
    gu = kernels.get("gemm_gate_up_swiglu")
    achieved = None
    if gu:
        avg_ms = gu["ms_total"] / gu["launches"]
        achieved = flops["gemm_gate_up_swiglu"] / (avg_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 1) if achieved else None,
                "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_sustained"], 4) if achieved else None,
                "traffic": recorded_traffic("gemm_gate_up_swiglu"), "traffic_unit": "bytes per launch (ncu dram read+write)",
                "kernel": "gemm_gate_up_swiglu: 832x28672x4096 tcgen05 GEMM with fused SwiGLU epilogue",
                "flops_per_launch": flops["gemm_gate_up_swiglu"], "avg_launch_ms": round(avg_ms, 5) if gu else None,
                "peak_source": f"{peaks['source']} bf16 sustained (kernel timed inside a long step)"}

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init weights N(0,0.02), uniform token ids)",
        "config": {"workload": WORKLOAD, "context_tokens": C, "query_tokens": fr.Q, "recomputed_rows": fr.ns,
                   "l2": "inputs larger than L2: 16 GB of weights and 671 MB of chunk K/V stream through every step",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "ttft_ms": round(ttft_ms, 3), "ttft_full_prefill_ms": round(full_ms, 3),
        "ttft_ratio_fused_over_full": round(ttft_ms / full_ms, 4),
        "ttft_method": (f"median of {n_ttft} requests, each alone and synchronised before and after (CUDA events on "
                        "the compute stream, first launch to first token on the host)"),
        "ttft_spread_ms": {"fused": [round(min(fused_ttfts), 3), round(max(fused_ttfts), 3)],
                           "full": [round(min(full_ttfts), 3), round(max(full_ttfts), 3)]},
        "back_to_back_ms": {"fused": round(ms_per_step, 4), "full": round(full_b2b_ms, 4),
                            "note": "steps enqueued back to back; consecutive requests overlap at their boundaries"},
        "ms_per_step_with_kernel_events": round(ms_with_events, 4),
        "e2e": {"value": round(world * C * args.steps / (e_ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ttft_ms": round(e_ms / args.steps, 3)},
        "gpu_launches": int(launches), "clocks": clk, "roofline": roofline, "kernels": kernels,
    }
    if selectors:
        out["selectors"] = selectors
    if dedupe:
        out["shared_chunks"] = dedupe
    if storage:
        out["storage_tier"] = storage
    out["host_link"] = measure_host_link(fr, device)
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(dm, fr, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ----------------------------------------------------------------- the oracle as CPU baseline

def _oracle_sample(weights_src, spec, req, ns, budget_s):
    """Times the oracle's fused path pieces on the 8B shapes and extrapolates one request.

    Sample: the critical-layer profile + top-N over the C context keys, one probe
    layer (64 query rows over the 80-anchor prefix) and one or more recompute
    layers (832 rows over the 5184-row fused cache), within `budget_s`.
    """
    from oracle import qcf_oracle as O
    om = O.OracleModel(weights_src, cache=False)
    rng = np.random.default_rng(0)
    C, Qn = req.chunk_len * req.n_chunks, req.query_len
    T = C + Qn
    Kc = rng.standard_normal((T, spec.n_kv_heads, spec.head_dim)).astype(np.float32)
    Vc = rng.standard_normal((T, spec.n_kv_heads, spec.head_dim)).astype(np.float32)
    q = (rng.standard_normal((Qn, spec.n_heads, spec.head_dim)) / math.sqrt(spec.head_dim)).astype(np.float32)
    W = om.layer(0)
    t0 = time.perf_counter()
    s = O.profile_scores(q, Kc[:C], 1.0 / math.sqrt(spec.head_dim))
    O.topn_select(s, O.num_selected(C, req.ratio_bp))
    t_select = time.perf_counter() - t0
    nA = req.n_chunks * req.n_anchor
    xp = rng.standard_normal((Qn, spec.d_model)).astype(np.float32)
    Kp, Vp = Kc[: nA + Qn].copy(), Vc[: nA + Qn].copy()
    t0 = time.perf_counter()
    O.layer_forward(xp, W, spec, C + np.arange(Qn), nA + np.arange(Qn), Kp, Vp)
    t_probe = time.perf_counter() - t0
    rows = np.concatenate([np.sort(rng.choice(C, ns - Qn, replace=False)), np.arange(C, T)])
    x = rng.standard_normal((ns, spec.d_model)).astype(np.float32)
    layers, t_layer = 0, 0.0
    while layers < 1 or (t_layer + t_probe + t_select < budget_s * 0.6 and layers < 3):
        t0 = time.perf_counter()
        O.layer_forward(x, W, spec, rows, rows, Kc, Vc)
        t_layer += time.perf_counter() - t0
        layers += 1
    ttft = t_select + req.crit_layer * t_probe + spec.n_layers * t_layer / layers
    sample = (f"oracle on the 8B shapes: profile+top-N over {C} keys, 1 probe layer (64 rows), {layers} recompute "
              f"layer(s) ({ns} rows over {T} cache rows); TTFT extrapolated to 16 probe + 32 recompute layers")
    return ttft, sample, t_select + t_probe + t_layer


def cpu_baseline(dm, fr, budget_s=20.0):
    spec, req = qd.LLAMA8B, qd.LLAMA8B_REQ

    class _Src:   # layer 0 of the device model's weights, unpacked, on the host
        def __init__(self):
            self.spec = spec

        def layer(self, l):
            t = dm.layer_tensors[l]
            Fp, F, d = dm.ffn_padded, spec.ffn, spec.d_model
            qw, kw = spec.q_width, spec.kv_width
            gu = t["w_gu"].view(Fp // 64, 2, 64, d)
            return {"wq": t["w_qkv"][:qw].cpu(), "wk": t["w_qkv"][qw:qw + kw].cpu(),
                    "wv": t["w_qkv"][qw + kw:].cpu(), "wo": t["w_o"].cpu(),
                    "wg": gu[:, 0].reshape(Fp, d)[:F].cpu(), "wu": gu[:, 1].reshape(Fp, d)[:F].cpu(),
                    "wd": t["w_down"][:, :F].cpu(), "g_attn": t["g_attn"].cpu(), "g_mlp": t["g_mlp"].cpu()}

    ttft, sample, measured = _oracle_sample(_Src(), spec, req, fr.ns, budget_s)
    cores = os.cpu_count()
    return {"value": round(fr.C / ttft, 2), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
            "extrapolated": True, "ttft_s_extrapolated": round(ttft, 2), "sample_s_measured": round(measured, 2),
            "threads": torch.get_num_threads()}


def run_reference(args):
    """The oracle as the reference arm, on the host cores, same metric and workload."""
    world, rank, _ = _dist_env()
    if rank != 0:
        return
    spec, req = qd.LLAMA8B, qd.LLAMA8B_REQ
    weights = qd.ModelWeights(spec)

    class _Layer0:
        def __init__(self):
            self.spec = spec

        def layer(self, l):
            return weights.layer(0)

    ns = qd.LLAMA8B_REQ.query_len + (req.ratio_bp * req.chunk_len * req.n_chunks + 9999) // 10000
    budget = max(5.0, 60.0 / max(1, args.steps + args.warmup))
    times, walls, sample = [], [], ""
    for i in range(args.warmup + args.steps):
        w0 = time.perf_counter()
        ttft, sample, _ = _oracle_sample(_Layer0(), spec, req, ns, budget)
        if i >= args.warmup:
            times.append(ttft)
            walls.append(time.perf_counter() - w0)
    ttft = statistics.mean(times)
    C = req.chunk_len * req.n_chunks
    v = C / ttft
    # a step is one bounded sample of the request (its pieces timed, the request's TTFT
    # extrapolated from them); ms_per_step is the sample's own wall time
    out = {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.mean(walls) * 1e3, 1),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "config": {"workload": WORKLOAD, "context_tokens": C},
           "extrapolated": True, "ttft_ms_extrapolated": round(ttft * 1e3, 1),
           "cpu_baseline": {"value": round(v, 2), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                            "sample": sample, "extrapolated": True},
           "e2e": {"value": round(v, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_oracle_e2e(args):
    """The oracle end to end on the host cores: the tiny request and the 8B-shaped request,
    fused (probe, profile, top-N, 32 recompute layers, LM head) and full prefill, each timed
    once.  Chunk K/V of the 8B request are the synthetic N(0,1) draws the parity tests use
    (chunk precompute is offline); weights are the seeded draws, converted to fp32 once
    before the timed calls."""
    from oracle import qcf_oracle as O
    res = {"oracle_e2e": {}, "cores": os.cpu_count(), "threads": torch.get_num_threads()}
    for name, spec, req, dev in (("tiny", qd.TINY, qd.TINY_REQ, "cpu"), ("llama8b", qd.LLAMA8B, qd.LLAMA8B_REQ, "cuda")):
        if dev == "cuda" and not torch.cuda.is_available():
            continue
        weights = qd.ModelWeights(spec, device=dev)
        om = O.OracleModel(weights, cache=True)
        t0 = time.perf_counter()
        for l in range(spec.n_layers):
            om.layer(l)
        om.embed_rows(np.zeros(1, np.int64))
        om.lm_head()
        prep = time.perf_counter() - t0
        ids = list(range(req.n_chunks))
        toks = [qd.chunk_tokens(c, req.chunk_len, spec.vocab) for c in ids]
        if name == "tiny":
            kv = [O.chunk_precompute(om, t) for t in toks]
        else:
            kv = []
            for c in ids:
                parts = [qd.synthetic_chunk_kv(spec, c, req.chunk_len, l, device=dev) for l in range(spec.n_layers)]
                kv.append({"K": O.as_f32(torch.stack([p["K"] for p in parts])),
                           "V": O.as_f32(torch.stack([p["V"] for p in parts]))})
        query = qd.query_tokens(0, req.query_len, spec.vocab)
        start = np.arange(req.n_chunks + 1) * req.chunk_len
        ctx = np.concatenate(toks)
        t0 = time.perf_counter()
        O.fused_prefill(om, kv, ctx, start, query, req.crit_layer, req.ratio_bp, req.n_anchor, keep_layers=False)
        t_fused = time.perf_counter() - t0
        t0 = time.perf_counter()
        O.full_prefill(om, np.concatenate([ctx, query]), keep_kv=False)
        t_full = time.perf_counter() - t0
        C = req.n_chunks * req.chunk_len
        res["oracle_e2e"][name] = {"fused_ttft_s": round(t_fused, 3), "full_prefill_s": round(t_full, 3),
                                   "context_tokens_per_s": round(C / t_fused, 2), "weight_prep_s": round(prep, 1),
                                   "context_tokens": C, "query_tokens": req.query_len}
        print(json.dumps({name: res["oracle_e2e"][name]}), flush=True)
        del om, weights, kv
    print(json.dumps(res), flush=True)


# ----------------------------------------------------------------- kernel sweep (profile + top-N, attention)


def profile_ceilings(ms, kbytes, flops, exps, peaks, exp_rate):
    """Fractions of the profile kernel against each ceiling (K read once from HBM; two
    tensor-core passes of Q K^T; two exp2 per score-row element); `bound` is the ceiling
    the kernel is closest to."""
    sec = ms * 1e-3
    fr = {"hbm": kbytes / sec / 1e9 / peaks["hbm_gbs"], "tensor": flops / sec / 1e12 / peaks["bf16"],
          "exp": exps / sec / exp_rate}
    bound = max(fr, key=fr.get)
    return {"bound": bound, "frac": round(fr[bound], 4), "hbm_gbs": round(kbytes / sec / 1e9, 1),
            "hbm_frac": round(fr["hbm"], 4), "tflops": round(flops / sec / 1e12, 1), "tensor_frac": round(fr["tensor"], 4),
            "exp_per_s": round(exps / sec / 1e12, 3), "exp_frac": round(fr["exp"], 4),
            "peaks": {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16"], "exp2_t_per_s": round(exp_rate / 1e12, 3)}}


def run_sweep(args):
    """Times profile+top-N and sparse causal attention on the kernel-sweep shapes
    (context 4k..128k, 64 query rows, 32 Q / 8 KV heads, head dim 128, 5..50 %
    selected, uniform or clustered), L2 flushed before every timed launch."""
    from rag_kv_cache_re_gb300 import qcf as Q
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    peaks = load_peaks()
    Hq, Hkv, D = qd.SWEEP_HEADS
    nq = qd.SWEEP_QUERY
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    reps = max(3, args.steps)
    exp_rate = Q.qcf_calibrate_exp2_rate(device)   # measured exp2/s of the special-function units
    print(json.dumps({"exp2_rate_per_s": exp_rate, "method": "qcf_calibrate_exp2_rate: 8 independent ex2.approx "
                      "chains per thread, 8 CTAs of 256 threads per SM, best of 2 timed launches"}), flush=True)

    def timed(fn):
        for _ in range(2):
            fn()
        ms = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        return statistics.median(ms)

    for C in qd.SWEEP_CONTEXTS:
        t = qd.sweep_tensors(C + nq, n_query=nq, device=str(device))
        K, V, q = t["K"], t["V"], t["Q"]
        Kc = K[:C]
        ms_prof = timed(lambda: Q.qcf_profile_scores(q, Kc, 1.0))
        scores = Q.qcf_profile_scores(q, Kc, 1.0)
        ws_topn = Q.workspace(Q._lib.lib().qcf_topn_select_workspace_size(C), device, "topn")
        kbytes = C * Hkv * D * 2
        exps = 2.0 * nq * Hq * C                 # two passes, one exp2 per score-row element each
        pflops = 2.0 * 2.0 * nq * Hq * C * D     # two passes of Q K^T
        for frac_bp in qd.SWEEP_FRACTIONS_BP:
            N = (frac_bp * C + 9999) // 10000
            ms_topn = timed(lambda: Q.qcf_topn_select_ws(scores, N, ws_topn))
            ms_topn_one = timed(lambda: Q.qcf_topn_select(scores, N))
            for pattern in ("uniform", "clusters"):
                pos = np.concatenate([qd.selected_indices(C, N, pattern), np.arange(C, C + nq)]).astype(np.int32)
                pos_d = torch.from_numpy(pos).to(device)
                qa = qd.normal_bf16((len(pos), Hq, D), 1.0 / math.sqrt(D), 9, str(device))
                ms_attn = timed(lambda: Q.qcf_sparse_causal_attn(qa, pos_d, K, V, 1.0))
                aflops = 4.0 * Hq * D * float(np.sum(pos.astype(np.float64) + 1))
                abytes = 2.0 * (C + nq) * Hkv * D * 2
                print(json.dumps({
                    "sweep": {"context": C, "selected_bp": frac_bp, "pattern": pattern, "N": int(N), "query_rows": nq},
                    "profile_topn_ms": round(ms_prof + ms_topn, 4), "profile_ms": round(ms_prof, 4),
                    "topn_ms": round(ms_topn, 4), "topn_one_cta_ms": round(ms_topn_one, 4),
                    "profile_roofline": profile_ceilings(ms_prof, kbytes, pflops, exps, peaks, exp_rate),
                    "attn_ms": round(ms_attn, 4),
                    "attn_roofline": {"bound": "tensor", "achieved": round(aflops / (ms_attn * 1e-3) / 1e12, 1),
                                      "peak": peaks["bf16"], "unit": "TFLOP/s",
                                      "frac": round(aflops / (ms_attn * 1e-3) / 1e12 / peaks["bf16"], 4),
                                      "hbm_gbs": round(abytes / (ms_attn * 1e-3) / 1e9, 1)},
                    "l2": "flushed (256 MB write) before every timed launch"}), flush=True)
                del qa, pos_d
        del t, K, V, q, scores
        torch.cuda.empty_cache()


def run_kernel(args):
    """Repeats one hot kernel on its bench shape (the target of the committed ncu captures):
    gate_up -- one 8B-shaped decoder layer over 832 recomputed rows of a 5184-row cache (its
    third GEMM launch is the gate/up projection with the SwiGLU epilogue);
    attention -- sparse causal attention at the 16k-context, 20 %-selected sweep point;
    attention8b -- sparse causal attention of one 8B recompute layer: 832 rows (768 selected of
    5120 context tokens, uniform, and the 64 query rows) over a 5184-row cache, scale 1/sqrt(128);
    profile -- critical-layer profiling at the 128k-context sweep point (64 query rows);
    topn -- top-N of the 128k profile scores at 15 % (the workspace entry point: cooperative grid)."""
    import dataclasses
    from rag_kv_cache_re_gb300 import model as M
    from rag_kv_cache_re_gb300 import qcf as Q
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    times = []
    if args.kernel == "gate_up":
        spec = dataclasses.replace(qd.LLAMA8B, n_layers=1, vocab=512)
        dm = M.DeviceModel(qd.ModelWeights(spec, device="cuda"), device, max_pos=8192)
        C, Qn, N = 5120, 64, 768
        rows = torch.as_tensor(np.concatenate([qd.selected_indices(C, N, "uniform"), np.arange(C, C + Qn)]).astype(np.int32),
                               device=device)
        x0 = torch.randn((N + Qn, spec.d_model), device=device)
        K = qd.normal_bf16((C + Qn, spec.n_kv_heads, spec.head_dim), 1.0, 71, "cuda")
        V = qd.normal_bf16((C + Qn, spec.n_kv_heads, spec.head_dim), 1.0, 72, "cuda")
        fn = lambda: Q.qcf_fused_layer_forward(dm, 0, x0.clone(), rows, rows, K, V)
    elif args.kernel == "attention8b":
        C, N = 5120, 768
        pos = torch.as_tensor(np.concatenate([qd.selected_indices(C, N, "uniform"), np.arange(C, C + 64)]).astype(np.int32),
                              device=device)
        t = qd.sweep_tensors(C + 64, n_query=len(pos), device="cuda")
        fn = lambda: Q.qcf_sparse_causal_attn(t["Q"], pos, t["K"], t["V"], 1.0 / math.sqrt(128))
    elif args.kernel in ("profile", "topn"):
        t = qd.sweep_tensors(131072, device="cuda")
        if args.kernel == "profile":
            fn = lambda: Q.qcf_profile_scores(t["Q"], t["K"], 1.0)
        else:
            sc = Q.qcf_profile_scores(t["Q"], t["K"], 1.0)
            ws_topn = Q.workspace(Q._lib.lib().qcf_topn_select_workspace_size(131072), device, "topn")
            fn = lambda: Q.qcf_topn_select_ws(sc, (1500 * 131072 + 9999) // 10000, ws_topn)
    else:
        Hq, Hkv, D = qd.SWEEP_HEADS
        C, N = 16384, 3277
        pos = torch.as_tensor(np.concatenate([qd.selected_indices(C, N, "uniform"), np.arange(C, C + 64)]).astype(np.int32),
                              device=device)
        t = qd.sweep_tensors(C + 64, n_query=len(pos), device="cuda")
        fn = lambda: Q.qcf_sparse_causal_attn(t["Q"], pos, t["K"], t["V"], 1.0)
    for _ in range(args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    print(json.dumps({"kernel": args.kernel, "ms": [round(v, 4) for v in times], "status": Q.qcf_query_status()}))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["qcf", "reference"], default="qcf")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--ttft-requests", type=int, default=20, help="synchronised single requests per TTFT median")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-selectors", action="store_true", help="skip timing the QCLast, QCAll and HKVD variants")
    ap.add_argument("--no-storage", action="store_true", help="skip timing the request served from files")
    ap.add_argument("--sweep", action="store_true", help="time the kernel-sweep shapes instead of the request")
    ap.add_argument("--oracle-e2e", action="store_true", help="time the oracle end to end (tiny and 8B, fused and full)")
    ap.add_argument("--kernel", choices=["gate_up", "attention", "attention8b", "profile", "topn"],
                    help="repeat one hot kernel (for ncu captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.oracle_e2e:
        run_oracle_e2e(args)
    elif args.sweep:
        run_sweep(args)
    elif args.kernel:
        run_kernel(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
