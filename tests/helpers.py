"""Shared test helpers: the parity gate and GPU run wrappers."""
import numpy as np

# Parity gate for float32 attention outputs against the f64 oracle:
#   max |gpu - oracle| <= 2e-5 over every element, and
#   max |gpu - oracle| / |oracle| <= 1e-4 over elements with |oracle| >= 0.2
#   (0.2 = 2e-5 / 1e-4, where the relative bound becomes the tighter one).
ATOL = 2e-5
RTOL = 1e-4
REL_FLOOR = ATOL / RTOL


def gate(gpu, ref, atol=ATOL, rtol=RTOL, where=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape
    assert np.all(np.isfinite(gpu)), f"{where}: non-finite GPU output"
    err = np.abs(gpu - ref)
    max_abs = float(err.max()) if err.size else 0.0
    big = np.abs(ref) >= REL_FLOOR
    max_rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    assert max_abs <= atol, f"{where}: max abs err {max_abs:.3e} > {atol:.1e}"
    assert max_rel <= rtol, f"{where}: max rel err {max_rel:.3e} > {rtol:.1e}"
    return max_abs, max_rel
