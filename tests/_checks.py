"""Comparison rules shared by the GPU parity tests.

Fused path (scores computed on the GPU in fp32 from fp8/bf16 inputs): every
score must lie within |d| <= 1e-3 * max(1, |s|) of the oracle's fp64 score, and
the selected set must equal the oracle's except for keys within that tolerance
of the oracle's k-th score:
  * every returned key has s >= s_k - tol(s_k)
  * every key with s > s_k + tol(s_k) is returned
which gives selected-value recall 1.0.  The row itself must be well formed:
min(topk, n) ascending, unique, in-range indices followed by -1.

Standalone top-k on given fp32 scores: byte-for-byte equal to the oracle.
"""
import numpy as np

REL_TOL = 1e-3


def tol(x):
    return REL_TOL * np.maximum(1.0, np.abs(x))


def check_row_shape(row, n, topk):
    m = min(topk, n)
    sel = row[:m]
    assert (row[m:] == -1).all(), "padding must be -1"
    assert (sel >= 0).all() and (sel < n).all(), "index out of the visible range"
    assert (np.diff(sel) > 0).all(), "indices must be ascending and unique"
    return sel


def check_fused_row(row, s_oracle, topk):
    """row: GPU indices of one row; s_oracle: fp64 scores of its visible keys."""
    n = len(s_oracle)
    sel = check_row_shape(np.asarray(row), n, topk)
    if n <= topk:
        assert len(sel) == n
        return 1.0
    kth = np.sort(s_oracle)[::-1][topk - 1]
    t = tol(kth)
    assert np.all(s_oracle[sel] >= kth - t), "a returned key is below the k-th score"
    must = np.flatnonzero(s_oracle > kth + t)
    assert np.isin(must, sel).all(), "a key clearly inside the top-k is missing"
    # selected-value recall against the oracle's own top-k values
    top_vals = np.sort(s_oracle)[::-1][:topk]
    got_vals = np.sort(s_oracle[sel])[::-1]
    return float(np.mean(np.abs(top_vals - got_vals) <= tol(top_vals)))


def check_scores(gpu, s_oracle):
    gpu = np.asarray(gpu, dtype=np.float64)
    d = np.abs(gpu - s_oracle)
    bad = d > tol(s_oracle)
    assert not bad.any(), (
        f"{bad.sum()} scores outside tolerance, worst |d|={d.max():.3g} "
        f"at {int(np.argmax(d))}")
    return float((d / np.maximum(1.0, np.abs(s_oracle))).max()) if d.size else 0.0
