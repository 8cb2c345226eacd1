"""Comparison rules between the CUDA path and the oracle (tolerances in one place).

* packing, Top-K and pooling of a given fp32 array: bit-exact;
* fp32 index scores: |s_gpu - s_ref| <= 1e-5 * sum_h |w_h| |q_h| |k_j| (the
  rounding-error scale of the sum; relative to |s| is ill-posed after ReLU
  cancellation);
* end-to-end Top-K sets: equal, except entries whose oracle score lies within
  that tolerance of the oracle's K-th score (both sides of a swap);
* attention: per (token, head) max|o - o_ref| / max|o_ref| <= 3e-3 against the
  float64 oracle on the same dequantised operands.
"""
import numpy as np

SCORE_RTOL = 1e-5
ATTN_RTOL = 3e-3
LSE_ATOL = 1e-3   # normaliser summed from fp32 or fp16-rounded P: relative difference <= 2^-11


def score_err(s_gpu, s_ref, cond):
    """max over entries of |s_gpu - s_ref| / cond (must be <= SCORE_RTOL)."""
    s_gpu = np.asarray(s_gpu, np.float64)
    s_ref = np.asarray(s_ref, np.float64)
    return float(np.max(np.abs(s_gpu - s_ref) / np.maximum(cond, 1e-30))) if len(s_ref) else 0.0


def check_topk_set(gpu_idx, gpu_cnt, ref_idx, scores_ref, cond, positions=None, k=None):
    """GPU selection vs oracle selection with near-threshold swaps allowed.

    scores_ref/cond are indexed like ``positions`` (None: by entry index).
    Returns the number of swapped entries.
    """
    gpu = np.asarray(gpu_idx[:gpu_cnt], np.int64)
    ref = np.asarray(ref_idx, np.int64)
    assert gpu_cnt == len(ref), f"count {gpu_cnt} != {len(ref)}"
    assert np.all(np.diff(gpu) > 0), "GPU selection is not strictly ascending"
    assert np.all(np.asarray(gpu_idx[gpu_cnt:]) == -1), "padding must be -1"
    diff = np.setxor1d(gpu, ref)
    if len(diff) == 0:
        return 0
    pos_of = (lambda e: e) if positions is None else (lambda e: int(np.searchsorted(positions, e)))
    s = np.asarray(scores_ref, np.float64)
    ref_pos = np.array([pos_of(e) for e in ref])
    kth = int(ref_pos[np.argmin(s[ref_pos])]) if len(ref_pos) else 0
    thr = s[kth]
    for e in diff:
        p = pos_of(e)
        if positions is not None:
            assert positions[p] == e, f"entry {e} is not a candidate"
        tol = SCORE_RTOL * (cond[p] + cond[kth])
        assert abs(s[p] - thr) <= tol, f"entry {e}: score {s[p]} vs threshold {thr} (tol {tol})"
    return len(diff)


def attn_err(O_gpu, O_ref):
    """max over heads of max|o - o_ref| / max|o_ref| (per (token, head) row)."""
    O_gpu = np.asarray(O_gpu, np.float64)
    O_ref = np.asarray(O_ref, np.float64)
    num = np.max(np.abs(O_gpu - O_ref), axis=-1)
    den = np.maximum(np.max(np.abs(O_ref), axis=-1), 1e-30)
    return float(np.max(num / den))
