"""Acceptance rules shared by the GPU parity tests (CUDA path vs the oracle)."""
import numpy as np

#: tie band for index sets: the oracle's k-th and (k+1)-th group scores may
#: differ by less than this (relative) before a choice between them is free
IDX_REL_BAND = 1e-4
O_MAX_ABS, O_MEAN_ABS = 2e-2, 2e-3
GRAD_REL_L2 = 3e-2
LSE_MAX_ABS = 1e-2
COV_BAND = 1e-4


def check_idx_row(gpu_row: np.ndarray, scores: np.ndarray, k: int, oracle_row: np.ndarray) -> str:
    """Returns '' if the GPU row is acceptable, else a reason.

    The row must hold k distinct ascending keys, contain every key scoring
    above tau (1 + band), hold none scoring below tau (1 - band) and agree
    with the oracle outside the band, tau being the oracle's k-th score.
    """
    g = np.asarray(gpu_row, dtype=np.int64)
    if g.shape != (k,):
        return f"length {g.shape}"
    if np.any(np.diff(g) <= 0):
        return "not strictly ascending"
    if g.min() < 0 or g.max() >= scores.shape[0]:
        return "index out of range"
    order = np.lexsort((np.arange(scores.shape[0]), -scores))
    tau = scores[order[k - 1]]
    band = IDX_REL_BAND * abs(tau)
    must = np.nonzero(scores > tau + band)[0]
    if not np.all(np.isin(must, g)):
        return "missing a key above the band"
    if np.any(scores[g] < tau - band):
        return "holds a key below the band"
    outside = np.abs(scores - tau) > band
    if not np.array_equal(np.isin(np.arange(scores.shape[0]), g) & outside,
                          np.isin(np.arange(scores.shape[0]), oracle_row) & outside):
        return "differs from the oracle outside the band"
    return ""


def check_kcov(curve: np.ndarray, k_gpu: int, mass: float = 0.9) -> str:
    """curve[k-1] = oracle C(k). Accept if C(k_gpu) >= mass - band and C(k_gpu - 1) < mass + band."""
    if not 1 <= k_gpu <= curve.shape[0]:
        return f"k_cov {k_gpu} out of range"
    if curve[k_gpu - 1] < mass - COV_BAND:
        return f"C({k_gpu}) = {curve[k_gpu - 1]:.6f} below {mass}"
    if k_gpu >= 2 and curve[k_gpu - 2] >= mass + COV_BAND:
        return f"C({k_gpu - 1}) = {curve[k_gpu - 2]:.6f} already reaches {mass}"
    return ""


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def o_errors(gpu: np.ndarray, ref: np.ndarray):
    d = np.abs(gpu - ref)
    return float(d.max()), float(d.mean())
