"""Sparse indexer, Top-K, hierarchical block pool and Reindex (steps a5-a9), in float64.

Test infrastructure only (see ``oracle/__init__.py``).

Sources (DeepSeek-V4.1 architecture analysis (blog.yuzhonghai.cloud), §02 "CSA2"):
* the indexer scores every causally visible compressed entry and the layer
  keeps the Top-512;
* modes: Full computes main KV, indexer K and Top-K itself; Reindex reuses
  the previous layer's global KV and indexer K and rescores them with its own
  indexer query; Reuse takes the Top-K indices unchanged;
* Hierarchical Sparse Indexer: after the Full layer's Top-512, blocks of 8
  positions are scored by the largest index score inside them, 2,048 blocks
  are kept (16,384 candidate positions), and Reindex layers search only there.

Readings where the pages are silent:
* score s_j = sum_h w_h * ReLU(q_h . k_j) over the indexer heads;
* entry j is visible to the token at raw position t iff 4j + 3 <= t;
* Top-K: the K largest scores, equal scores ordered by lower index, all
  visible entries when fewer than K are visible; output is the set in
  ascending index order, padded with -1, plus its count;
* blocks are aligned (block b = positions 8b..8b+7); a block's score is the
  maximum over its visible positions; blocks without a visible position are
  not candidates; if fewer than 2,048 blocks are visible all of them are kept;
  equal block scores are ordered by lower block id;
* scores that are zero compare equal regardless of sign.
"""
from __future__ import annotations

import numpy as np


def n_visible(n_entries: int, t: int) -> int:
    """Number of entries visible at raw position t: j visible iff 4j+3 <= t."""
    return int(max(0, min(n_entries, (t + 1) // 4)))


def index_scores(q: np.ndarray, w: np.ndarray, K: np.ndarray) -> np.ndarray:
    """Step a5 for one query token: s_j = sum_h w_h * max(0, q_h . k_j).

    q [Hi, Di], w [Hi], K [n, Di] (the visible entries) -> fp32 scores [n]
    (accumulated in float64, rounded once).
    """
    q = np.asarray(q, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    dots = K @ q.T                      # [n, Hi]
    s = np.maximum(dots, 0.0) @ w       # [n]
    return s.astype(np.float32)


def score_condition(q: np.ndarray, w: np.ndarray, K: np.ndarray) -> np.ndarray:
    """Scale of the rounding error of s_j: sum_h |w_h| * |q_h| * |k_j| (float64)."""
    qn = np.linalg.norm(np.asarray(q, dtype=np.float64), axis=1)
    kn = np.linalg.norm(np.asarray(K, dtype=np.float64), axis=1)
    return np.outer(kn, qn) @ np.abs(np.asarray(w, dtype=np.float64))


def topk(scores: np.ndarray, k: int) -> np.ndarray:
    """Step a6: indices of the k highest scores (ties -> lower index), ascending.

    A full stable sort on (score descending, index ascending).  Returns an
    int64 array of min(k, n) indices in ascending order.
    """
    s = np.asarray(scores, dtype=np.float64)
    n = s.shape[0]
    order = np.lexsort((np.arange(n), -s))  # last key is primary
    return np.sort(order[:min(k, n)])


def pad(idx: np.ndarray, k: int) -> np.ndarray:
    out = np.full(k, -1, dtype=np.int64)
    out[:len(idx)] = idx
    return out


def block_scores(scores: np.ndarray, block: int = 8) -> np.ndarray:
    """Block max over the visible positions (the scores given): [ceil(n / block)]."""
    s = np.asarray(scores, dtype=np.float64)
    n = s.shape[0]
    nb = -(-n // block)
    return np.array([np.max(s[b * block:min(n, (b + 1) * block)]) for b in range(nb)],
                    dtype=np.float64)


def block_pool(scores: np.ndarray, n_blocks: int = 2048, block: int = 8) -> np.ndarray:
    """Step a7: ids of the n_blocks blocks with the largest block max, ascending."""
    return topk(block_scores(scores, block), n_blocks)


def pool_positions(pool: np.ndarray, n_vis: int, block: int = 8) -> np.ndarray:
    """Visible positions of the pooled blocks, ascending."""
    pos = (np.asarray(pool, dtype=np.int64).reshape(-1, 1) * block
           + np.arange(block).reshape(1, -1)).reshape(-1)
    return pos[pos < n_vis]


def full_select(q, w, K_all, t, k, hierarchical=False, n_blocks=2048, block=8):
    """Full mode for one query token: score all visible entries, Top-K, optional pool.

    Returns dict(idx=ascending int64 indices, scores=fp32 [n_vis], pool=block ids or None).
    """
    nv = n_visible(K_all.shape[0], t)
    s = index_scores(q, w, K_all[:nv])
    idx = topk(s, k)
    pool = block_pool(s, n_blocks, block) if hierarchical else None
    return {"idx": idx, "scores": s, "pool": pool, "n_vis": nv}


def reindex_select(q, w, K_all, t, k, pool, block=8):
    """Reindex mode for one query token: score only the pool's visible positions, Top-K.

    The scores are those of index_scores at the pooled positions; the Top-K
    ranks them with ties broken by the lower entry index.
    """
    nv = n_visible(K_all.shape[0], t)
    pos = pool_positions(pool, nv, block)
    s = index_scores(q, w, K_all[pos]) if len(pos) else np.zeros(0, np.float32)
    sel = topk(s, k)              # positions within pos, which is ascending
    return {"idx": pos[sel], "scores": s, "positions": pos}


def reuse_select(idx_in: np.ndarray) -> np.ndarray:
    """Reuse mode (step a9): the previous layer's indices, unchanged."""
    return np.array(idx_in, copy=True)
