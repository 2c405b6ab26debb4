"""Acceptance checks shared by the GPU parity tests.

The bar for BF16 I/O with FP32 accumulation: per element
|gpu - oracle| <= 2e-2 + 2e-2 |oracle|, and relative Frobenius error <= 5e-3.
"""

import numpy as np

ATOL = 2e-2
RTOL = 2e-2
FROB = 5e-3


def assert_parity(gpu, ref, atol=ATOL, rtol=RTOL, frob=FROB, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, f"{what}: shape {gpu.shape} vs {ref.shape}"
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    err = np.abs(gpu - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(ref))), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: gpu={gpu[i]} oracle={ref[i]}")
    denom = np.linalg.norm(ref)
    rel = np.linalg.norm(gpu - ref) / denom if denom > 0 else np.linalg.norm(gpu)
    assert rel <= frob, f"{what}: relative Frobenius error {rel:.3e} > {frob}"
    return float(err.max()), float(rel)
