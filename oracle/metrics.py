"""Error metrics (oracle; test infrastructure only).

"miniTE technical report", section 2.3: for a reference vector x and a decoded
vector x_hat of n elements, relative L2 = ||x_hat - x|| / ||x||,
SNR = 20 log10(||x|| / ||x_hat - x||) in dB, MAE = (1/n) sum |x_hat_j - x_j|.
"""
from __future__ import annotations

import numpy as np


def rel_l2(x_hat, x) -> float:
    x = np.asarray(x, dtype=np.float64).ravel()
    d = np.asarray(x_hat, dtype=np.float64).ravel() - x
    return float(np.linalg.norm(d) / np.linalg.norm(x))


def snr_db(x_hat, x) -> float:
    x = np.asarray(x, dtype=np.float64).ravel()
    d = np.asarray(x_hat, dtype=np.float64).ravel() - x
    return float(20.0 * np.log10(np.linalg.norm(x) / np.linalg.norm(d)))


def mae(x_hat, x) -> float:
    x = np.asarray(x, dtype=np.float64).ravel()
    return float(np.mean(np.abs(np.asarray(x_hat, dtype=np.float64).ravel() - x)))


def rel_frobenius(got, ref) -> float:
    """||got - ref||_F / ||ref||_F (the GEMM parity measure)."""
    return rel_l2(got, ref)


def max_abs_err(got, ref) -> float:
    return float(np.max(np.abs(np.asarray(got, dtype=np.float64)
                               - np.asarray(ref, dtype=np.float64))))


def within_gemm_tolerance(got, ref, rel=1e-3, elem=1e-2):
    """Relative Frobenius error <= rel and max |got - ref| <= elem * max |ref|."""
    ref = np.asarray(ref, dtype=np.float64)
    rf = rel_frobenius(got, ref) if np.any(ref) else float(np.max(np.abs(got)))
    mx = max_abs_err(got, ref)
    bound = elem * float(np.max(np.abs(ref))) if ref.size else 0.0
    return (rf <= rel and mx <= bound), rf, mx, bound
