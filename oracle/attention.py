"""Gathered sparse MQA attention over the selected entries plus the FP8 window (a10-a11).

Test infrastructure only (see ``oracle/__init__.py``).

Sources:
* fewer KV heads (many query heads share one KV head), attention over the
  Top-K entries: DeepSeek-V4.1 architecture analysis (blog.yuzhonghai.cloud),
  §02 "CSA2";
* FP4 main KV is dequantised back before attention; the sliding-window KV of
  the last n_win = 128 raw tokens is kept in FP8: same page, §03.

Readings where the pages are silent:
* K = V = the dequantised 512-d latent (one shared KV head);
* one softmax over {selected compressed entries} U {window tokens
  max(0, t-W+1) .. t}; a key present in both sets is counted twice;
* logits q_h . k * tau with tau = 1/sqrt(d); no attention sink;
* operands: Q in bf16, main-KV entries dequantised exactly, window tokens
  dequantised to bf16(fp32(e4m3 * scale)); the oracle works in float64 on
  exactly those values.
"""
from __future__ import annotations

import numpy as np


def softmax_attention(Q: np.ndarray, keys: np.ndarray, tau: float):
    """o_h = sum_i softmax_i(q_h . k_i * tau) k_i  (values = keys). Returns (O, lse).

    Q [Hq, d], keys [n, d] -> O [Hq, d] float64, lse [Hq] (natural log of the
    softmax denominator, including the max shift).
    """
    Q = np.asarray(Q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    logits = (Q @ keys.T) * tau                  # [Hq, n]
    m = np.max(logits, axis=1, keepdims=True)
    p = np.exp(logits - m)
    l = np.sum(p, axis=1, keepdims=True)
    O = (p @ keys) / l
    return O, (m + np.log(l)).reshape(-1)


def window_positions(t: int, W: int) -> np.ndarray:
    """Raw positions of the sliding window seen by the token at t: max(0, t-W+1) .. t."""
    return np.arange(max(0, t - W + 1), t + 1, dtype=np.int64)


def sparse_attention(Q, kv_sel: np.ndarray, swa: np.ndarray, tau: float):
    """Step a11 for one query token: one softmax over selected entries then window tokens.

    kv_sel [n_sel, d] dequantised main-KV rows, swa [n_win, d] dequantised
    window rows.  Rows with no selected entry attend to the window only.
    """
    keys = np.concatenate([np.asarray(kv_sel, np.float64).reshape(-1, swa.shape[1]),
                           np.asarray(swa, np.float64)], axis=0)
    return softmax_attention(Q, keys, tau)


def dense_causal_attention(Q: np.ndarray, kv_all: np.ndarray, t: int,
                           swa_all: np.ndarray, swa_pos: np.ndarray, W: int, tau: float):
    """Independent dense form used to pin sparse_attention.

    Attends from the token at t over *every* cached entry and every window row
    with a 0/1 mask (entry j allowed iff 4j+3 <= t; window row at position p
    allowed iff t-W < p <= t), computing the normaliser with log-sum-exp.
    """
    Q = np.asarray(Q, dtype=np.float64)
    keys = np.concatenate([np.asarray(kv_all, np.float64), np.asarray(swa_all, np.float64)])
    j = np.arange(kv_all.shape[0])
    allowed = np.concatenate([4 * j + 3 <= t,
                              (np.asarray(swa_pos) > t - W) & (np.asarray(swa_pos) <= t)])
    logits = Q @ keys.T * tau
    logits = np.where(allowed[None, :], logits, -np.inf)
    lse = np.logaddexp.reduce(logits, axis=1)
    w = np.exp(logits - lse[:, None])
    return w @ keys, lse
