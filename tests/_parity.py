"""Comparison helpers for GPU-vs-oracle parity tests."""
import numpy as np


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
