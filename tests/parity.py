"""Shared parity helpers for the GPU tests (oracle comparison, tolerances)."""
import numpy as np

# GEMV tolerance: relative L2 error <= 1e-3 and per element |err| <= 2e-3 * sum_j |w_ij x_j|
REL_L2 = 1e-3
ELEM = 2e-3


def check_gemv(y_gpu: np.ndarray, y_ref: np.ndarray, a_ref: np.ndarray, what: str = "") -> None:
    y_gpu = np.asarray(y_gpu, np.float64).reshape(y_ref.shape)
    err = np.abs(y_gpu - y_ref)
    assert np.isfinite(y_gpu).all(), f"{what}: non-finite output"
    denom = np.linalg.norm(y_ref)
    rel = np.linalg.norm(y_gpu - y_ref) / denom if denom > 0 else np.linalg.norm(y_gpu)
    assert rel <= REL_L2, f"{what}: relative L2 {rel:.3e} > {REL_L2}"
    bad = err > ELEM * a_ref + 1e-30
    assert not bad.any(), f"{what}: {bad.sum()} elements exceed 2e-3*sum|wx| (worst {(err / (a_ref + 1e-30)).max():.3e})"
