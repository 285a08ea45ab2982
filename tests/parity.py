"""Comparison helpers shared by the GPU parity tests (no method arithmetic).

Tolerances:
  * floats (attention output, self-conditioning): per row,
    max|gpu - ref| / max|ref| <= 2e-2 (bf16 inputs, fp32 accumulation);
  * log-sum-exp: |gpu - ref| <= 1e-2 absolute;
  * conf = exp(max logit - lse), so its relative error is bounded by the
    lse tolerance: |gpu - ref| / ref <= 1e-2;
  * integers (Philox draws, re-noised tokens, copies): bit-exact;
  * decisions (argmax, conf < threshold): identical, except at positions the
    oracle flags (top-2 probability gap, or |conf - threshold|, below 1e-3),
    which must be fewer than 0.5% of positions.
"""
import numpy as np

ROW_REL = 2e-2
LSE_ABS = 1e-2
CONF_REL = 1e-2
FLAG = 1e-3
FLAG_BUDGET = 0.005


def row_rel_err(gpu, ref):
    gpu = np.asarray(gpu, np.float64).reshape(ref.shape[0], -1)
    ref = np.asarray(ref, np.float64).reshape(ref.shape[0], -1)
    num = np.abs(gpu - ref).max(axis=1)
    den = np.maximum(np.abs(ref).max(axis=1), 1e-30)
    return num / den


def assert_rows_close(gpu, ref, tol=ROW_REL, what="rows"):
    err = row_rel_err(gpu, ref)
    worst = int(np.argmax(err))
    assert np.isfinite(err).all() and err.max() <= tol, f"{what}: max row rel err {err.max():.3e} at row {worst}"
    return float(err.max())


def decision_flags(ref, threshold):
    """Positions whose decision floating point may legitimately flip."""
    conf = np.asarray(ref["conf"], np.float64)
    near_thr = np.abs(conf - threshold) < FLAG
    kept = conf >= threshold
    gap = (conf - np.asarray(ref["p2"], np.float64)) < FLAG
    return near_thr | (kept & gap)


def logit_gap_flags(ref):
    """Rows whose argmax is decided by a logit gap below 1e-3 (relative)."""
    m = np.asarray(ref["max_logit"], np.float64)
    l2 = np.asarray(ref["l2"], np.float64)
    return (m - l2) < FLAG * np.maximum(1.0, np.abs(m))
