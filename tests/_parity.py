"""Comparison helpers for GPU-vs-oracle parity tests."""
import numpy as np


def assert_close(got, ref, atol, rtol, what=""):
    """|got - ref| <= atol + rtol*|ref| elementwise (allclose semantics)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
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
