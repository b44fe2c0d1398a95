"""Why the bf16 hidden-state tolerance scales its absolute term with the tensor's RMS (CPU).

The CUDA path keeps the residual stream in fp32 but feeds every GEMM bf16
operands: the RMSNorm output h, the projected q/k/v, the attention output o and
the SwiGLU activation are rounded to bf16 (round to nearest even), and the
fused cache stores K/V as bf16.  This test rebuilds one decoder layer at the
Llama-3-8B layer shape (d 4096, 32 Q / 8 KV heads, head dim 128, FFN 14336)
over the 8B request's 832 recomputed rows of a 5184-row cache, with exactly
those roundings and no other change, and compares it with the fp32/fp64 oracle:

* under the plain allclose bound |got - ref| <= 2e-2 + 2e-2 |ref| this
  emulation FAILS: rounding a GEMM operand moves every output of its row by
  about 2^-9 of the row's scale, whatever the element's own value, so elements
  near zero in a tensor of RMS above 1 exceed a fixed 2e-2;
* with the absolute term 2e-2 * max(1, RMS(ref)) it passes.

So a kernel that rounds no more than its operands' storage format demands
cannot meet the unscaled bound, and the scaled one is the tightest bound of
that form the storage format allows.  The emulation shares no code with the
CUDA path; it calls the oracle's own layer pieces and adds the roundings.
"""
import dataclasses

import numpy as np
import pytest

import qcfdata as qd
from oracle import qcf_oracle as O
from _bf16_emulation import layer as emulated_layer

F32, F64 = np.float32, np.float64


def excess(got, ref, atol, rtol, rms_scaled):
    """max over elements of |got-ref| / (atol' + rtol |ref|); <= 1 passes."""
    got, ref = np.asarray(got, F64), np.asarray(ref, F64)
    if rms_scaled:
        atol = atol * max(1.0, float(np.sqrt(np.mean(ref * ref))))
    return float(np.max(np.abs(got - ref) / (atol + rtol * np.abs(ref))))


@pytest.mark.slow
def test_bf16_operand_rounding_needs_the_rms_scaled_bound():
    spec = dataclasses.replace(qd.LLAMA8B, n_layers=1, vocab=512)
    W = O.OracleModel(qd.ModelWeights(spec), cache=False).layer(0)
    C, T, N = 5120, 5184, 768
    rows = np.concatenate([qd.selected_indices(C, N, "uniform"), np.arange(C, T)]).astype(np.int64)
    rng = np.random.default_rng(42)
    x = rng.standard_normal((len(rows), spec.d_model)).astype(F32)
    K0 = O.as_f32(qd.normal_bf16((T, spec.n_kv_heads, spec.head_dim), 1.0, 43))
    V0 = O.as_f32(qd.normal_bf16((T, spec.n_kv_heads, spec.head_dim), 1.0, 44))

    Kr, Vr = K0.copy(), V0.copy()
    ref = O.layer_forward(x, W, spec, rows, rows, Kr, Vr)
    Ke, Ve = K0.copy(), V0.copy()
    emu = emulated_layer(x, W, spec, rows, rows, Ke, Ve)

    pairs = {"x after the layer": (emu, ref), "fresh K": (Ke[rows], Kr[rows]), "fresh V": (Ve[rows], Vr[rows])}
    strict = {k: excess(g, r, 2e-2, 2e-2, False) for k, (g, r) in pairs.items()}
    scaled = {k: excess(g, r, 2e-2, 2e-2, True) for k, (g, r) in pairs.items()}
    print("strict", strict, "scaled", scaled)
    assert max(strict.values()) > 1.0, f"the unscaled bound already holds for bf16 operands: {strict}"
    assert max(scaled.values()) <= 1.0, f"bf16 operand rounding alone exceeds the scaled bound: {scaled}"


def test_sampled_rows_equal_the_whole_layer():
    """oracle_layer_rows (every row's fresh K/V first, then the layer on a subset) gives the
    subset's rows of the whole layer: rows interact only through the cache."""
    from _parity import oracle_layer_rows
    spec = dataclasses.replace(qd.TINY, n_layers=1)
    W = O.OracleModel(qd.ModelWeights(spec)).layer(0)
    C, T = 96, 104
    rows = np.concatenate([qd.selected_indices(C, 20, "uniform"), np.arange(C, T)]).astype(np.int64)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((len(rows), spec.d_model)).astype(F32)
    K0 = rng.standard_normal((T, spec.n_kv_heads, spec.head_dim)).astype(F32)
    V0 = rng.standard_normal((T, spec.n_kv_heads, spec.head_dim)).astype(F32)
    Kw, Vw = K0.copy(), V0.copy()
    whole = O.layer_forward(x, W, spec, rows, rows, Kw, Vw)
    smp = np.array([0, 3, 19, 20, 27])
    Ks, Vs = K0.copy(), V0.copy()
    part = oracle_layer_rows(x, W, spec, rows, Ks, Vs, smp)
    np.testing.assert_allclose(part, whole[smp], atol=1e-6, rtol=1e-6)
    np.testing.assert_allclose(Ks, Kw, atol=1e-6, rtol=1e-6)   # BLAS blocking differs with the row count
    np.testing.assert_allclose(Vs, Vw, atol=1e-6, rtol=1e-6)


@pytest.mark.slow
def test_bf16_storage_alone_exceeds_the_scaled_bound_at_the_34b_shape():
    """At the Yi-34B layer shape (d 7168, 56 Q / 8 KV heads, FFN 20480, the 34B request's
    20608-row cache; 512 recomputed context rows and the 128 query rows, to keep the CPU
    time down) the hidden states after one layer have an
    RMS near 5.5, and bf16 storage of the operands alone departs from the fp32 oracle by
    more than even the RMS-scaled bound: past one layer at that scale, or many layers at
    any scale, the only attainable bound is the error of bf16 storage itself."""
    from _parity import oracle_layer_rows
    import _bf16_emulation as E
    spec = dataclasses.replace(qd.YI34B, n_layers=1, vocab=512)
    W = O.OracleModel(qd.ModelWeights(spec), cache=False).layer(0)
    C, T, N = 20480, 20608, 512
    rows = np.concatenate([qd.selected_indices(C, N, "uniform"), np.arange(C, T)]).astype(np.int64)
    rng = np.random.default_rng(50)
    x = rng.standard_normal((len(rows), spec.d_model)).astype(F32)
    K0 = O.as_f32(qd.normal_bf16((T, spec.n_kv_heads, spec.head_dim), 1.0, 60))
    V0 = O.as_f32(qd.normal_bf16((T, spec.n_kv_heads, spec.head_dim), 1.0, 61))
    smp = np.unique(np.concatenate([np.arange(N, len(rows)), rng.choice(N, 128, replace=False)]))
    Kr, Vr = K0.copy(), V0.copy()
    ref = oracle_layer_rows(x, W, spec, rows, Kr, Vr, smp)
    Ke, Ve = K0.copy(), V0.copy()
    emu = oracle_layer_rows(x, W, spec, rows, Ke, Ve, smp, kv_projection=E.kv_projection, layer=E.layer)
    scaled = excess(emu, ref, 2e-2, 2e-2, True)
    print("34B shape, bf16 storage vs oracle, scaled excess", scaled, "x RMS", float(np.sqrt(np.mean(ref.astype(F64) ** 2))))
    assert scaled > 1.0
    assert excess(Ke[rows], Kr[rows], 2e-2, 2e-2, True) <= 1.0   # one projection deep: within the bound
