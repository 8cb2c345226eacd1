"""Compression of new tokens into MXFP4 KV entries (steps a1-a4), in float64.

Test infrastructure only (see ``oracle/__init__.py``).

Sources:
* 4:1 sequence compression, one entry per 4 consecutive tokens:
  DeepSeek-V4.1 architecture analysis (blog.yuzhonghai.cloud), §02 "CSA2"
  ("compress the sequence dimension, every m tokens into one entry"), and the
  DeepSeek V4 review (wmrh.cn), §2.2 (4 tokens -> 1 entry); the same review,
  §2.1, describes the compression as a pure linear projection.
* RMSNorm over the whole 512-d latent, RoPE that preserves the norm, and
  quantisation after RoPE: DeepSeek-V4.1 architecture analysis, §03.

Readings where the pages are silent (each stated in the library header too):
* the map is linear without bias on the token-major concatenation
  [h_4j; h_4j+1; h_4j+2; h_4j+3]; a trailing partial group makes no entry;
* RMSNorm: x = c / sqrt(mean(c^2) + eps) * gamma over all d channels;
* RoPE rotates the last r channels with rotate-half pairing (i, i + r/2),
  inv_freq_i = base^(-2i/r), at the position of the entry's last token, 4j+3;
* the indexer key of a new entry is a second linear map W_idx of the same
  concatenation, stored in the indexer dtype (bf16, or fp32 when so configured).
"""
from __future__ import annotations

import numpy as np

from . import formats


def concat_groups(hidden: np.ndarray) -> np.ndarray:
    """[T, H] hidden states -> [T//4, 4H]: row j = [h_4j; h_4j+1; h_4j+2; h_4j+3]."""
    hidden = np.asarray(hidden, dtype=np.float64)
    T, H = hidden.shape
    n = T // 4
    out = np.empty((n, 4 * H), dtype=np.float64)
    for j in range(n):
        for k in range(4):
            out[j, k * H:(k + 1) * H] = hidden[4 * j + k]
    return out


def compress(hidden: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Step a1: c_j = W @ concat(h_4j..h_4j+3); float64 product, rounded to fp32.

    W is [d, 4H] (row o produces output channel o).
    """
    cat = concat_groups(hidden)
    c = cat @ np.asarray(W, dtype=np.float64).T
    return c.astype(np.float32).astype(np.float64)


def rmsnorm(c: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """Step a2 (first half): x = c / sqrt(mean(c^2) + eps) * gamma, row-wise; fp32 result."""
    c = np.asarray(c, dtype=np.float64)
    ms = np.mean(c * c, axis=-1, keepdims=True)
    x = c / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)
    return x.astype(np.float32).astype(np.float64)


def rope(x: np.ndarray, positions: np.ndarray, r: int, base: float) -> np.ndarray:
    """Step a2 (second half): rotate the last r channels of each row; fp32 result.

    For pair i < r/2 the channels (d-r+i, d-r+i+r/2) are rotated by the angle
    pos * base^(-2i/r).
    """
    x = np.array(x, dtype=np.float64)
    d = x.shape[-1]
    half = r // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = base ** (-2.0 * i / r)
    ang = np.asarray(positions, dtype=np.float64).reshape(-1, 1) * inv_freq.reshape(1, -1)
    cos, sin = np.cos(ang), np.sin(ang)
    a = x[:, d - r:d - half].copy()
    b = x[:, d - half:].copy()
    x[:, d - r:d - half] = a * cos - b * sin
    x[:, d - half:] = a * sin + b * cos
    return x.astype(np.float32).astype(np.float64)


def entry_position(j) -> np.ndarray:
    """Raw position used for entry j's rotation and visibility: its last token, 4j+3."""
    return 4 * np.asarray(j, dtype=np.int64) + 3


def norm_rope_pack(latent: np.ndarray, entry_ids: np.ndarray, gamma, eps, r, base):
    """Steps a2-a3 on given latent rows: returns (post-RoPE fp32 x, codes, scales)."""
    x = rmsnorm(latent, gamma, eps)
    x = rope(x, entry_position(entry_ids), r, base)
    codes, scales = formats.mxfp4_pack(x.astype(np.float32))
    return x, codes, scales


def norm_rope_pack_fp8(latent: np.ndarray, entry_ids: np.ndarray, gamma, eps, r, base):
    """Steps a2 and the V4-style FP8 main-KV pack on given latent rows: returns
    (post-RoPE fp32 x, E4M3 codes [n, d], fp32 scales [n]).

    The same RMSNorm and RoPE as the MXFP4 entries; the row is then packed by the
    FP8 rule of the sliding window (one scale per row, amax / 448).  The DeepSeek V4
    review and the V4.1 analysis (§03, V4.1's FP4 main KV halves V4's FP8 one)
    describe this format only as V4's; it is kept to compare the two.
    """
    x = rmsnorm(latent, gamma, eps)
    x = rope(x, entry_position(entry_ids), r, base)
    codes, scales = formats.fp8_pack(x.astype(np.float32))
    return x, codes, scales


def compress_pack(hidden, W, gamma, eps, r, base, first_entry: int, W_idx=None,
                  idx_dtype: str = "bf16", kv_format: str = "mxfp4"):
    """Steps a1-a4 for one sequence's new tokens [T, H] (T a multiple of 4 or not).

    Returns a dict with the fp32 latent c, the post-RoPE x, the MXFP4 codes and
    scales of entries first_entry .. first_entry + T//4 - 1, and (if W_idx is
    given) their indexer keys.
    """
    c = compress(hidden, W)
    ids = first_entry + np.arange(c.shape[0])
    pack = norm_rope_pack_fp8 if kv_format == "fp8" else norm_rope_pack
    x, codes, scales = pack(c, ids, gamma, eps, r, base)
    out = {"c": c, "x": x, "codes": codes, "scales": scales, "entry_ids": ids}
    if W_idx is not None:
        k = concat_groups(hidden) @ np.asarray(W_idx, dtype=np.float64).T
        k32 = k.astype(np.float32)
        out["idx_k"] = formats.bf16_round(k32) if idx_dtype == "bf16" else k32.astype(np.float64)
    return out
