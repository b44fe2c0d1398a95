"""Comparison helpers for GPU-vs-oracle parity tests."""
import numpy as np

from oracle import qcf_oracle as O


def assert_close(got, ref, atol, rtol, what="", rms_scaled=False):
    """|got - ref| <= atol + rtol*|ref| elementwise (allclose semantics).

    rms_scaled: the absolute term is atol * max(1, RMS(ref)).  Used for bf16
    hidden states and K/V: rounding a GEMM operand to bf16 (relative 2^-9)
    perturbs every output of the row by an amount set by the row's scale, not by
    the element's own value, so elements near zero in a tensor of RMS s see
    errors of order 2^-9 * s.  A numpy forward that rounds the same operands to
    bf16 departs from the fp32 oracle exactly as much as the kernels do.
    """
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if rms_scaled and ref.size:
        atol = atol * max(1.0, float(np.sqrt(np.mean(ref * ref))))
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref) - (atol + rtol * np.abs(ref))
    worst = np.unravel_index(np.argmax(err), err.shape) if err.size else None
    assert err.size == 0 or err.max() <= 0, (
        f"{what}: max excess {err.max():.3e} at {worst}: got {got[worst]:.6g} ref {ref[worst]:.6g}")


def assert_same_selection(got_idx, ref_values, k, tie_tol, what=""):
    """got_idx (the kernel's k indices) must equal the oracle's top-k of ref_values
    (ties to the lower index), except for swaps among candidates whose oracle
    values lie within tie_tol of the oracle's k-th value."""
    ref_values = np.asarray(ref_values, dtype=np.float64)
    got = np.sort(np.asarray(got_idx, dtype=np.int64))
    assert len(got) == k, f"{what}: {len(got)} indices, want {k}"
    assert len(np.unique(got)) == k, f"{what}: duplicate indices"
    if k == 0:
        return
    order = np.argsort(-ref_values, kind="stable")
    ref = np.sort(order[:k])
    if np.array_equal(got, ref):
        return
    kth = ref_values[order[k - 1]]
    sym = set(got.tolist()) ^ set(ref.tolist())
    bad = [j for j in sym if abs(ref_values[j] - kth) > tie_tol]
    assert not bad, f"{what}: selection differs beyond ties at {bad[:8]} (kth={kth:.6g})"


def error_stats(got, ref):
    """(max-abs, RMS) of got - ref."""
    d = np.asarray(got, np.float64) - np.asarray(ref, np.float64)
    if d.size == 0:
        return 0.0, 0.0
    return float(np.max(np.abs(d))), float(np.sqrt(np.mean(d * d)))


def assert_close_bf16_floor(got, ref, emu, what="", atol=2e-2, rtol=2e-2, rms_factor=1.25, max_factor=2.0):
    """The RMS-scaled allclose bound of assert_close, or, where it fails, the error
    bf16 storage alone forces as the bound.

    emu is the oracle's arithmetic with every GEMM operand and cache entry stored as
    bf16 (tests/_bf16_emulation.py).  Through many layers, or through one layer whose
    activations are large (the 34B and 70B shapes), that unavoidable error exceeds the
    fixed bound; the kernel's error must then stay within rms_factor times the
    emulation's RMS error over the tensor and within max_factor times its largest
    element's error (the extreme of millions of rounding errors is the noisier
    statistic, so it gets the wider factor)."""
    try:
        assert_close(got, ref, atol, rtol, what=what, rms_scaled=True)
        return "allclose"
    except AssertionError as strict_fail:
        g_max, g_rms = error_stats(got, ref)
        e_max, e_rms = error_stats(emu, ref)
        assert np.all(np.isfinite(np.asarray(got, np.float64))), f"{what}: non-finite values"
        assert g_max <= max_factor * e_max and g_rms <= rms_factor * e_rms, (
            f"{what}: beyond the allclose bound ({strict_fail}) and beyond the bf16-storage error "
            f"(x{rms_factor} RMS, x{max_factor} max): "
            f"max {g_max:.4g} vs {e_max:.4g}, RMS {g_rms:.4g} vs {e_rms:.4g}")
        return f"bf16 floor: max {g_max:.4g} vs {e_max:.4g}, RMS {g_rms:.4g} vs {e_rms:.4g}"


def oracle_layer_rows(x, W, spec, rows, Kc, Vc, smp, kv_projection=O.kv_projection, layer=O.layer_forward):
    """One layer of recompute for the rows x at cache rows `rows`, output only for the
    subset `smp` (indices into x): every row's fresh K/V is written into the cache first
    (kv_projection), then the layer runs on the subset over that cache.  Rows do not
    interact except through the cache, so the subset's outputs are those of the whole
    layer.  Kc / Vc are updated in place."""
    k, v = kv_projection(x, W, spec, rows)
    Kc[rows] = k
    Vc[rows] = v
    return layer(x[smp], W, spec, rows[smp], rows[smp], Kc, Vc)
