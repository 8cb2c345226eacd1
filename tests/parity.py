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


# ---- bytes packed after a GEMM (compression, CED projection, window replay) ---------------
#
# A packed byte decided from a GEMM's fp32 sums can differ from the oracle's
# (float64 sums) only where the oracle's pre-quantisation value lies within the
# computation's error bound of a rounding boundary, and then by one grid step.
# The bound is propagated from the GEMM outputs to each decision:
#   GEMM output      |c_gpu - c_ref| <= GEMM_KAPPA * sum_i |a_i b_i|  (fp32 accumulation
#                    of up to 16,384 products in tensor-core blocks and split-K partials;
#                    the compression GEMM of the 4,096-token chunk, K = 16,384 in 6 splits,
#                    measured at most 2^-22.3 of that sum against float64 on a GB300)
#   RMSNorm          |dx_i| <= (|gamma_i| tau_i + |x_i| rms(tau)) / (rho - rms(tau))
#   RoPE             a rotated channel takes the bound of both channels of its pair
#   fp32 roundings   + FP32_ROUND * |x| (sum of squares, sqrt, products, rotation)
# Every packed value must be the rounding of some value within the bound of the
# oracle's pre-quantisation value: it lies between the roundings of value - bound
# and value + bound (rounding is monotonic).  Where the bound is below half a grid
# step that is the oracle's code, or one step away where the value lies within the
# bound of the rounding boundary between the two (a sign change only where it lies
# within the bound of zero); only grid steps finer than the bound (E4M3 subnormals
# at the bottom of a row's range) can move further.  A scale code is checked
# against amax/6; the group's E2M1 codes then against the GPU's own scale.

GEMM_KAPPA = 2.0 ** -20
FP32_ROUND = 2.0 ** -20


def gemm_error_bound(a, w):
    """Per-output bound GEMM_KAPPA * sum_i |a_i| |w_i| of a product a @ w.T ([n, K] x [m, K])."""
    return GEMM_KAPPA * (np.abs(np.asarray(a, np.float64)) @ np.abs(np.asarray(w, np.float64)).T)


def latent_error_bound(c_ref, tau_c, gamma, eps, r, x_ref):
    """Bound on |x_gpu - x_ref| of RMSNorm + RoPE rows, given |c_gpu - c_ref| <= tau_c."""
    c_ref = np.asarray(c_ref, np.float64)
    tau_c = np.asarray(tau_c, np.float64)
    d = c_ref.shape[-1]
    rho = np.sqrt(np.mean(c_ref * c_ref, axis=-1, keepdims=True) + eps)
    t_rho = np.sqrt(np.mean(tau_c * tau_c, axis=-1, keepdims=True))
    xn = np.abs(c_ref / rho * np.asarray(gamma, np.float64))
    tx = (np.abs(np.asarray(gamma, np.float64)) * tau_c + xn * t_rho) / np.maximum(rho - t_rho, 1e-30)
    if r:
        half = r // 2
        a, b = slice(d - r, d - half), slice(d - half, d)
        pair = tx[..., a] + tx[..., b]
        tx[..., a] = pair
        tx[..., b] = pair
    return tx + FP32_ROUND * (np.abs(np.asarray(x_ref, np.float64)) + xn)


def _e2m1_nibbles(codes):
    codes = np.asarray(codes, np.uint8)
    c4 = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.uint8)
    c4[..., 0::2] = codes & 0xF
    c4[..., 1::2] = codes >> 4
    return c4


def _in_rounding_interval(code_g, v, tv, table, encode, sign_bit):
    """Codes code_g (int array) against values v with bounds tv (same shape, in code units):
    True where the code's value lies between the values of encode(v - tv) and
    encode(v + tv), and its sign bit is that of some value in [v - tv, v + tv]."""
    lo = table[encode((v - tv).astype(np.float32)).astype(np.int64)]
    hi = table[encode((v + tv).astype(np.float32)).astype(np.int64)]
    val = table[code_g]
    neg = (code_g & sign_bit) != 0
    sign_ok = np.where(neg, v - tv <= 0, v + tv >= 0)
    return (val >= lo) & (val <= hi) & sign_ok


def check_mxfp4_after_gemm(codes_g, scales_g, x_ref, tau_x):
    """GPU MXFP4 bytes of rows [n, d] against the oracle's post-RoPE fp32 rows x_ref.

    Returns (number of scale flips, number of code flips); raises on any other difference.
    """
    from oracle import formats as F
    x_ref = np.asarray(x_ref, np.float64)
    tau_x = np.asarray(tau_x, np.float64)
    n, d = x_ref.shape
    G = d // 16
    sg = np.asarray(scales_g, np.uint8).reshape(n, G)
    xg = x_ref.reshape(n, G, 16)
    tg = tau_x.reshape(n, G, 16)
    u = (np.max(np.abs(xg), axis=2).astype(np.float32) / np.float32(6.0)).astype(np.float32).astype(np.float64)
    s_exp = F.e4m3_encode_array(u)
    flip = sg != s_exp
    if flip.any():
        tau_u = np.max(tg, axis=2)[flip] / 6.0 + FP32_ROUND * u[flip]
        ok = _in_rounding_interval(sg[flip].astype(np.int64), u[flip], tau_u, F.E4M3_TABLE, F.e4m3_encode_array,
                                   0x80)
        assert ok.all(), (f"scales outside the roundings of the bound: gpu {sg[flip][~ok][:5]}, oracle "
                          f"{s_exp[flip][~ok][:5]}, amax/6 {u[flip][~ok][:5]}, bound {tau_u[~ok][:5]}")
    # codes against the GPU's own scale of each group
    s_val = F.E4M3_TABLE[sg].astype(np.float32)
    safe = np.where(s_val == 0, np.float32(1.0), s_val).astype(np.float32)
    q = (xg.astype(np.float32) / safe[:, :, None]).astype(np.float32)
    c_exp = np.where((s_val == 0)[:, :, None], 0, F.e2m1_encode_array(q)).astype(np.uint8)
    c_gpu = _e2m1_nibbles(codes_g).reshape(n, G, 16)
    diff = c_gpu != c_exp
    if diff.any():
        assert not (diff & (s_val == 0)[:, :, None]).any(), "a group with a zero scale has non-zero codes"
        sb = np.broadcast_to(s_val[:, :, None].astype(np.float64), xg.shape)[diff]
        ok = _in_rounding_interval(c_gpu[diff].astype(np.int64), xg[diff] / sb, tg[diff] / sb, F.E2M1_TABLE,
                                   F.e2m1_encode_array, 8)
        assert ok.all(), (f"codes outside the roundings of the bound: gpu {c_gpu[diff][~ok][:5]}, oracle "
                          f"{c_exp[diff][~ok][:5]}, x/scale {(xg[diff] / sb)[~ok][:5]}, bound "
                          f"{(tg[diff] / sb)[~ok][:5]}")
    return int(flip.sum()), int(diff.sum())


def check_keys_after_gemm(k_gpu, k_exact, tau_k, dtype):
    """Indexer keys stored by the GPU against the oracle's float64 projection.

    bf16: the stored value must be the bf16 rounding of some value within the bound of
    the exact one, i.e. lie between the roundings of exact - bound and exact + bound
    (rounding is monotonic).  Where the bound is below half a bf16 step this is the
    oracle's rounding, or one step away where the exact value lies within the bound of
    the midpoint; only keys smaller than about 2^8 bounds can move further.  fp32:
    within the bound.  Returns the number of keys that differ from the oracle's rounding."""
    from oracle import formats as F
    k_gpu = np.asarray(k_gpu, np.float64)
    k_exact = np.asarray(k_exact, np.float64)
    tau = np.asarray(tau_k, np.float64) + FP32_ROUND * np.abs(k_exact)
    if dtype != "bf16":
        err = np.abs(k_gpu - k_exact)
        assert np.all(err <= tau), f"fp32 keys beyond the GEMM bound: {err[err > tau][:5]}"
        return 0
    lo = F.bf16_round((k_exact - tau).astype(np.float32))
    hi = F.bf16_round((k_exact + tau).astype(np.float32))
    ok = (k_gpu >= lo) & (k_gpu <= hi)
    assert ok.all(), (f"bf16 keys outside the roundings of the bound: gpu {k_gpu[~ok][:5]}, exact "
                      f"{k_exact[~ok][:5]}, bound {tau[~ok][:5]}")
    return int(np.sum(k_gpu != F.bf16_round(k_exact.astype(np.float32))))


def check_fp8_after_gemm(codes_g, scales_g, x_ref, tau_x):
    """GPU FP8 window rows [n, d] (codes) and [n] (scales) against the oracle's fp32 rows.

    scale = amax / 448: within the row's bound / 448 of the oracle's; codes against
    E4M3(x / the GPU's scale) under the rounding-interval rule above.  Returns the
    number of codes that differ."""
    from oracle import formats as F
    x_ref = np.asarray(x_ref, np.float64)
    tau_x = np.asarray(tau_x, np.float64)
    sg = np.asarray(scales_g, np.float32)
    s_ref = (np.max(np.abs(x_ref), axis=1).astype(np.float32) / np.float32(448.0)).astype(np.float64)
    t_s = np.max(tau_x, axis=1) / 448.0 + FP32_ROUND * s_ref
    bad = np.abs(sg - s_ref) > t_s
    assert not bad.any(), f"window scales beyond the bound: gpu {sg[bad][:5]}, oracle {s_ref[bad][:5]}"
    safe = np.where(sg == 0, np.float32(1.0), sg).astype(np.float32)
    q = (x_ref.astype(np.float32) / safe[:, None]).astype(np.float32)
    c_exp = np.where((sg == 0)[:, None], 0, F.e4m3_encode_array(q)).astype(np.uint8)
    cg_all = np.asarray(codes_g, np.uint8)
    diff = cg_all != c_exp
    if diff.any():
        s_b = np.broadcast_to(sg[:, None].astype(np.float64), x_ref.shape)[diff]
        ok = _in_rounding_interval(cg_all[diff].astype(np.int64), x_ref[diff] / s_b, tau_x[diff] / s_b,
                                   F.E4M3_TABLE, F.e4m3_encode_array, 0x80)
        assert ok.all(), (f"FP8 codes outside the roundings of the bound: gpu {cg_all[diff][~ok][:5]}, oracle "
                          f"{c_exp[diff][~ok][:5]}, x/scale {(x_ref[diff] / s_b)[~ok][:5]}")
    return int(diff.sum())
