"""Seeded synthetic inputs shared by the CUDA path, the oracle, the tests and the bench.

This module only draws numbers: model shapes, random-init weights, token ids,
synthetic K/V/Q tensors, selected-index patterns and request layouts.  It holds
none of the method's arithmetic (no normalisation, rotation, attention,
scoring or selection), so that the oracle and the CUDA path share nothing but
their inputs.

Distributions follow the workloads of the QCFuse / CacheBlend pages: random-init
Llama-style decoders with weights N(0, 0.02), uniform token ids, requests of
many retrieved chunks of a few hundred to ~1k tokens followed by a short query,
and, for the kernel sweep, K, V ~ N(0, 1) and Q ~ N(0, 1)/sqrt(128).

Every weight and every stored K/V value is rounded to bfloat16 (round to
nearest even) where it is drawn, so both sides consume identical values.
Seeds: weights 0, tokens 1, sweep tensors 2, selection indices 3, the
shared-chunk permutation 4.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

SEED_WEIGHTS = 0
SEED_TOKENS = 1
SEED_SWEEP = 2
SEED_SELECT = 3
SEED_PERMUTE = 4


@dataclasses.dataclass(frozen=True)
class ModelSpec:
    """Shape of a Llama-style decoder (RMSNorm, RoPE, GQA attention, SwiGLU)."""

    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    theta: float = 1e4
    eps: float = 1e-5

    @property
    def q_width(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_width(self) -> int:
        return self.n_kv_heads * self.head_dim


@dataclasses.dataclass(frozen=True)
class RequestSpec:
    """One request: retrieved chunks (by id, in retrieval order) then a query."""

    chunk_len: int
    n_chunks: int
    query_len: int
    crit_layer: int
    ratio_bp: int          # recompute ratio in basis points (1500 = 15 %)
    n_anchor: int


TINY = ModelSpec("tiny", n_layers=2, d_model=64, n_heads=4, n_kv_heads=4,
                 head_dim=16, ffn=172, vocab=256)
LLAMA8B = ModelSpec("llama3-8b-shape", n_layers=32, d_model=4096, n_heads=32,
                    n_kv_heads=8, head_dim=128, ffn=14336, vocab=128256)
YI34B = ModelSpec("yi-34b-shape", n_layers=60, d_model=7168, n_heads=56,
                  n_kv_heads=8, head_dim=128, ffn=20480, vocab=64000)
LLAMA70B = ModelSpec("llama-70b-shape", n_layers=80, d_model=8192, n_heads=64,
                     n_kv_heads=8, head_dim=128, ffn=28672, vocab=32000)

TINY_REQ = RequestSpec(chunk_len=32, n_chunks=3, query_len=8, crit_layer=1,
                       ratio_bp=1500, n_anchor=2)
LLAMA8B_REQ = RequestSpec(chunk_len=512, n_chunks=10, query_len=64, crit_layer=16,
                          ratio_bp=1500, n_anchor=8)
YI34B_REQ = RequestSpec(chunk_len=1024, n_chunks=20, query_len=128, crit_layer=30,
                        ratio_bp=1000, n_anchor=8)
LLAMA70B_REQ = RequestSpec(chunk_len=512, n_chunks=35, query_len=64, crit_layer=40,
                           ratio_bp=1500, n_anchor=8)

SWEEP_CONTEXTS = (4096, 16384, 65536, 131072)
SWEEP_FRACTIONS_BP = (500, 1000, 2000, 5000)
SWEEP_QUERY = 64
SWEEP_HEADS = (32, 8, 128)     # H_q, H_kv, D


def _gen(seed: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _mix(*parts: int) -> int:
    """Deterministic 63-bit seed from a tuple of small integers (splitmix-style)."""
    h = 0x9E3779B97F4A7C15
    for p in parts:
        h ^= (int(p) + 0x632BE59BD9B4E019 + ((h << 6) & 0xFFFFFFFFFFFFFFFF) + (h >> 2))
        h &= 0xFFFFFFFFFFFFFFFF
        h = (h * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        h ^= h >> 31
    return h & 0x7FFF_FFFF_FFFF_FFFF


def normal_bf16(shape: Sequence[int], std: float, seed: int, device: str = "cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32 and rounded to bf16 (RNE), on `device`."""
    t = torch.randn(tuple(shape), generator=_gen(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


# Weight tensors of one decoder layer, in nn.Linear layout [out_features][in_features].
LAYER_MATRICES = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def layer_weight_shapes(spec: ModelSpec) -> Dict[str, tuple]:
    d, F = spec.d_model, spec.ffn
    return {
        "wq": (spec.q_width, d), "wk": (spec.kv_width, d), "wv": (spec.kv_width, d),
        "wo": (d, spec.q_width), "wg": (F, d), "wu": (F, d), "wd": (d, F),
    }


class ModelWeights:
    """Random-init weights N(0, 0.02) in bf16, generated per tensor from its own seed.

    Any tensor can be regenerated alone (the oracle streams large models layer by
    layer).  RMSNorm gains are 1.  The LM head is untied from the embedding.
    Values are reproducible per (seed, device type); CPU and CUDA draws differ.
    """

    def __init__(self, spec: ModelSpec, seed: int = SEED_WEIGHTS, device: str = "cpu",
                 std: float = 0.02):
        self.spec, self.seed, self.device, self.std = spec, seed, device, std

    def _draw(self, shape, *key) -> torch.Tensor:
        return normal_bf16(shape, self.std, _mix(self.seed, *key), self.device)

    def layer(self, l: int) -> Dict[str, torch.Tensor]:
        shapes = layer_weight_shapes(self.spec)
        out = {name: self._draw(shapes[name], 1, l, i) for i, name in enumerate(LAYER_MATRICES)}
        ones = torch.ones(self.spec.d_model, dtype=torch.bfloat16, device=self.device)
        out["g_attn"] = ones
        out["g_mlp"] = ones.clone()
        return out

    def embed(self) -> torch.Tensor:
        return self._draw((self.spec.vocab, self.spec.d_model), 2)

    def lm_head(self) -> torch.Tensor:
        return self._draw((self.spec.vocab, self.spec.d_model), 3)

    def final_norm(self) -> torch.Tensor:
        return torch.ones(self.spec.d_model, dtype=torch.bfloat16, device=self.device)


def token_ids(n: int, vocab: int, stream: int, seed: int = SEED_TOKENS) -> np.ndarray:
    """Uniform token ids in [0, vocab); `stream` separates chunks and queries."""
    g = _gen(_mix(seed, stream))
    return torch.randint(0, vocab, (n,), generator=g, dtype=torch.int64).numpy().astype(np.int32)


def chunk_tokens(chunk_id: int, length: int, vocab: int) -> np.ndarray:
    """Tokens of a retrieved chunk; the same chunk id always gives the same tokens."""
    return token_ids(length, vocab, stream=1_000_000 + int(chunk_id))


def query_tokens(request: int, length: int, vocab: int) -> np.ndarray:
    return token_ids(length, vocab, stream=2_000_000 + int(request))


def request_layout(req: RequestSpec, chunk_ids: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """Chunk boundaries of a request (chunks in retrieval order, then the query)."""
    ids = list(range(req.n_chunks)) if chunk_ids is None else [int(c) for c in chunk_ids]
    lens = np.full(len(ids), req.chunk_len, dtype=np.int32)
    start = np.zeros(len(ids) + 1, dtype=np.int32)
    start[1:] = np.cumsum(lens)
    return {"chunk_ids": np.asarray(ids, dtype=np.int32), "chunk_start": start,
            "context_len": int(start[-1]), "query_len": req.query_len}


def shared_chunk_requests(n_chunks: int = 35, share_frac: float = 0.70,
                          seed: int = SEED_PERMUTE) -> List[np.ndarray]:
    """Two requests of `n_chunks` chunk ids that share round-half-up(share_frac*n) ids.

    Request A uses ids 0..n-1 in a seeded random order; request B takes the shared
    ids (the first ones of A's order) plus fresh ids, in its own seeded order.
    """
    n_shared = int(math.floor(share_frac * n_chunks + 0.5))
    g = _gen(seed)
    a = torch.randperm(n_chunks, generator=g).numpy()
    shared = a[:n_shared]
    fresh = np.arange(n_chunks, n_chunks + (n_chunks - n_shared))
    b_ids = np.concatenate([shared, fresh])
    b = b_ids[torch.randperm(n_chunks, generator=g).numpy()]
    return [a.astype(np.int32), b.astype(np.int32)]


def sweep_tensors(C: int, n_query: int = SWEEP_QUERY, Hq: int = 32, Hkv: int = 8, D: int = 128,
                  seed: int = SEED_SWEEP, device: str = "cpu") -> Dict[str, torch.Tensor]:
    """K, V ~ N(0,1) [C][Hkv][D] and Q ~ N(0,1)/sqrt(D) [n_query][Hq][D], all bf16."""
    return {
        "K": normal_bf16((C, Hkv, D), 1.0, _mix(seed, C, 1), device),
        "V": normal_bf16((C, Hkv, D), 1.0, _mix(seed, C, 2), device),
        "Q": normal_bf16((n_query, Hq, D), 1.0 / math.sqrt(D), _mix(seed, C, 3), device),
    }


def selected_indices(C: int, N: int, pattern: str, seed: int = SEED_SELECT) -> np.ndarray:
    """N distinct ascending indices in [0, C): 'uniform' or 'clusters' (8 contiguous runs)."""
    g = _gen(_mix(seed, C, N, 0 if pattern == "uniform" else 1))
    if N <= 0:
        return np.zeros(0, dtype=np.int32)
    if pattern == "uniform":
        idx = torch.randperm(C, generator=g)[:N].numpy()
        return np.sort(idx).astype(np.int32)
    if pattern != "clusters":
        raise ValueError(pattern)
    n_cl = min(8, N)
    per = -(-N // n_cl)
    lens = [per] * n_cl
    lens[-1] = N - per * (n_cl - 1)
    free = C - N
    cuts = np.sort(torch.randint(0, free + 1, (n_cl,), generator=g).numpy())
    out, prev_end, prev_cut = [], 0, 0
    for k in range(n_cl):
        start = prev_end + (int(cuts[k]) - prev_cut)
        out.append(np.arange(start, start + lens[k]))
        prev_end, prev_cut = start + lens[k], int(cuts[k])
    return np.concatenate(out).astype(np.int32)


def synthetic_chunk_kv(spec: ModelSpec, chunk_id: int, length: int, layer: int,
                       device: str = "cpu", seed: int = SEED_SWEEP) -> Dict[str, torch.Tensor]:
    """Stand-in precomputed chunk K/V ~ N(0,1) [length][H_kv][D] bf16 for large shapes."""
    shape = (length, spec.n_kv_heads, spec.head_dim)
    return {"K": normal_bf16(shape, 1.0, _mix(seed, 7, chunk_id, layer, 1), device),
            "V": normal_bf16(shape, 1.0, _mix(seed, 7, chunk_id, layer, 2), device)}


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round an fp32 array to the nearest bf16 value (ties to even), returned as fp32."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()
