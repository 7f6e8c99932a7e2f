"""Helpers shared by the GPU tests: build/load the library, upload arrays, tolerances."""
import numpy as np
import pytest

FP32_TOL = 1e-3   # rtol = atol for float32 paths
LOW_TOL = 2e-2    # rtol = atol for bfloat16 and 4-bit paths


def lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from weight_streaming_gemv_token_gb300 import build

    build.build()
    import weight_streaming_gemv_token_gb300 as W

    W.library()
    return W


def dev(a):
    from weight_streaming_gemv_token_gb300.decoder import to_device

    return to_device(a)


def close(got, ref, tol, what=""):
    """|got - ref| <= tol + tol * |ref| elementwise (the oracle is the reference)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref)
    bad = err > tol + tol * np.abs(ref)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tol {tol}; first at {i}: "
                             f"got {got.ravel()[i]!r} ref {ref.ravel()[i]!r}; max err {err.max():.3e}")
    return float(err.max()) if err.size else 0.0


def accumulation_bound(Wm, x, n_terms):
    """Float32 accumulation error bound for y = W x: 2 n u sum|w x| (u = 2^-24)."""
    from oracle import widen

    return 2.0 * n_terms * 2.0 ** -24 * (np.abs(widen(Wm)) @ np.abs(widen(x))) + 1e-30
