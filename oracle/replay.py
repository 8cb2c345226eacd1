"""SWA Bounded Replay: a layer's sliding window rebuilt from its last tokens, in float64.

Test infrastructure only (see ``oracle/__init__.py``).

Source: DeepSeek-V4.1 architecture analysis (blog.yuzhonghai.cloud), §03
"SWA Bounded Replay".  The window KV is not kept in the persistent cache; it
is rebuilt by replaying only the last n_win = 128 raw tokens, which cuts the
state short: a token early in the replay sees fewer window rows than the
exact state would give it, and the pages accept that the rebuilt state
differs.  The same section keeps the window KV in FP8, and the window keys
share one softmax with the main-KV entries (§02-§03), so a window row lives
in the same latent space as a compressed entry.

Readings where the pages are silent (stated in the library header too):
* a window row is the latent of one raw token, x_t = RoPE_t(RMSNorm(W_swa h_t)):
  W_swa [d, H] linear without bias on that token's hidden state, the RMSNorm of
  the main KV (gain gamma, eps), RoPE at the token's own raw position t (not an
  entry position 4j+3), then the per-token FP8 pack of the window;
* the replayed token at raw position p sees the window rows at raw positions
  max(p0, p - W + 1) .. p, p0 being the first replayed position (the rebuilt
  window holds nothing before it).
"""
from __future__ import annotations

import numpy as np

from . import compress, formats


def project(hidden: np.ndarray, W_swa: np.ndarray) -> np.ndarray:
    """c_t = W_swa h_t for every row of hidden [n, H]; float64 product rounded to fp32."""
    c = np.asarray(hidden, dtype=np.float64) @ np.asarray(W_swa, dtype=np.float64).T
    return c.astype(np.float32).astype(np.float64)


def window_rows(hidden, W_swa, gamma, eps, r, base, pos0: int):
    """Window rows of the replayed tokens at raw positions pos0 .. pos0 + n - 1.

    Returns a dict with the fp32 projection c, the post-RoPE x and the FP8
    codes [n, d] and scales [n] of each row.
    """
    c = project(hidden, W_swa)
    x = compress.rmsnorm(c, gamma, eps)
    x = compress.rope(x, pos0 + np.arange(c.shape[0], dtype=np.int64), r, base)
    codes, scales = formats.fp8_pack(x.astype(np.float32))
    return {"c": c, "x": x, "codes": codes, "scales": scales}


def replay_window_positions(t: int, W: int, p0: int) -> np.ndarray:
    """Raw positions of the rebuilt window seen by the replayed token at t: max(p0, t-W+1) .. t."""
    return np.arange(max(p0, t - W + 1), t + 1, dtype=np.int64)
