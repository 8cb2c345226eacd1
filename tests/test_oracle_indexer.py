"""Pins of oracle/indexer.py: brute force, library routines, the pages' pool constants."""
import numpy as np
import pytest
import torch

from golden_io import load
from oracle import indexer as I

PAGE = load("page_constants.json")


def _brute_topk(s, k):
    """Entry i is selected iff fewer than k entries rank before it (higher, or equal and lower)."""
    s = [float(v) for v in s]
    n = len(s)
    sel = []
    for i in range(n):
        rank = sum(1 for j in range(n) if s[j] > s[i] or (s[j] == s[i] and j < i))
        if rank < k:
            sel.append(i)
    return np.array(sel, dtype=np.int64)


def test_scores_closed_forms():
    g = np.random.default_rng(0)
    q = g.normal(0, 1, (1, 16))
    K = g.normal(0, 1, (50, 16))
    s = I.index_scores(q, np.array([1.0]), K)
    assert np.allclose(s, np.maximum(K @ q[0], 0).astype(np.float32))
    assert np.all(s >= 0) and (s == 0).any()                # the ReLU clips
    s_neg = I.index_scores(q, np.array([-2.0]), K)
    assert np.allclose(s_neg, -2 * s, rtol=1e-6)


def test_scores_brute_force_and_torch():
    g = np.random.default_rng(1)
    Hi, Di, n = 4, 8, 30
    q, w, K = g.normal(0, 1, (Hi, Di)), g.normal(0, 1, Hi), g.normal(0, 1, (n, Di))
    s = I.index_scores(q, w, K)
    for j in range(n):
        acc = 0.0
        for h in range(Hi):
            dot = sum(q[h, i] * K[j, i] for i in range(Di))
            acc += w[h] * (dot if dot > 0 else 0.0)
        assert abs(s[j] - acc) <= 1e-6 * (1 + abs(acc))
    ref = torch.einsum("hd,nd->nh", torch.from_numpy(q), torch.from_numpy(K)).relu() @ torch.from_numpy(w)
    assert np.allclose(s, ref.numpy().astype(np.float32), rtol=1e-6, atol=1e-6)
    cond = I.score_condition(q, w, K)
    assert np.all(np.abs(s) <= cond * (1 + 1e-6))


def test_visibility_rule():
    # entry j is visible at t iff 4j + 3 <= t
    assert I.n_visible(100, 2) == 0
    assert I.n_visible(100, 3) == 1
    assert I.n_visible(100, 6) == 1
    assert I.n_visible(100, 7) == 2
    assert I.n_visible(100, 10 ** 6) == 100
    for t in range(0, 60):
        nv = I.n_visible(1000, t)
        assert all(4 * j + 3 <= t for j in range(nv))
        assert not (4 * nv + 3 <= t)


@pytest.mark.parametrize("n,k,levels", [(40, 7, 1000), (40, 7, 3), (25, 30, 5), (60, 60, 2), (1, 1, 1)])
def test_topk_brute_force(n, k, levels):
    g = np.random.default_rng(n * 100 + k)
    s = g.integers(0, levels, n).astype(np.float32) - levels // 2
    got = I.topk(s, k)
    assert np.array_equal(got, _brute_topk(s, k))
    assert len(got) == min(k, n) and np.all(np.diff(got) > 0)


def test_topk_all_equal_takes_lowest_indices_and_signed_zeros_tie():
    assert np.array_equal(I.topk(np.zeros(10, np.float32), 4), np.arange(4))
    s = np.array([0.0, -0.0, 0.0, -0.0, -1.0], dtype=np.float32)
    assert np.array_equal(I.topk(s, 2), [0, 1])


def test_topk_matches_torch_on_distinct_values():
    g = torch.Generator().manual_seed(2)
    s = torch.randperm(5000, generator=g).to(torch.float32) * 0.37 - 900.0
    assert torch.unique(s).numel() == 5000
    ref = torch.sort(torch.topk(s, 512).indices).values.numpy()
    assert np.array_equal(I.topk(s.numpy(), PAGE["top_k"]["value"]), ref)


def _walk_pool(s, n_blocks, block):
    """Walk entries in (score desc, index asc) order collecting distinct blocks."""
    order = np.lexsort((np.arange(len(s)), -np.asarray(s, np.float64)))
    seen = []
    for j in order:
        b = j // block
        if b not in seen:
            seen.append(b)
            if len(seen) == n_blocks:
                break
    return np.sort(np.array(seen, dtype=np.int64))


def test_block_pool_by_entry_walk():
    g = np.random.default_rng(3)
    for n, nb in [(200, 7), (203, 7), (50, 100), (8 * 2048 + 5, 2048)]:
        s = g.integers(0, 40, n).astype(np.float32)          # many ties
        assert np.array_equal(I.block_pool(s, nb, 8), _walk_pool(s, nb, 8))


def test_pool_size_and_topk_inclusion():
    nb, bs, K = PAGE["pool_blocks"]["value"], PAGE["pool_block_size"]["value"], PAGE["top_k"]["value"]
    g = np.random.default_rng(4)
    n = 3 * nb * bs + 5                                       # ragged last block
    s = g.normal(0, 1, n).astype(np.float32)
    pool = I.block_pool(s, nb, bs)
    pos = I.pool_positions(pool, n, bs)
    if pool[-1] != (n - 1) // bs:
        assert len(pos) == nb * bs == PAGE["pool_positions"]["value"]
    assert len(pool) == nb
    assert set(I.topk(s, K)).issubset(set(pos))               # Full Top-512 is inside the pool


def test_pool_keeps_all_blocks_when_few_are_visible():
    s = np.random.default_rng(5).normal(0, 1, 100).astype(np.float32)
    pool = I.block_pool(s, 2048, 8)
    assert np.array_equal(pool, np.arange(13))
    assert np.array_equal(I.pool_positions(pool, 100, 8), np.arange(100))


def test_reindex_with_full_query_reproduces_full_selection():
    g = np.random.default_rng(6)
    Hi, Di, n = 4, 16, 40000
    K = g.normal(0, 1, (n, Di))
    q, w = g.normal(0, 1, (Hi, Di)), g.normal(0, 1, Hi)
    t = 4 * n + 10
    full = I.full_select(q, w, K, t, 512, hierarchical=True, n_blocks=2048, block=8)
    re = I.reindex_select(q, w, K, t, 512, full["pool"], 8)
    assert np.array_equal(re["idx"], full["idx"])
    assert len(re["positions"]) == PAGE["pool_positions"]["value"]
    # a different query searches only inside the pool
    q2 = g.normal(0, 1, (Hi, Di))
    re2 = I.reindex_select(q2, w, K, t, 512, full["pool"], 8)
    assert set(re2["idx"]).issubset(set(re2["positions"]))


def test_causal_selection_and_truncation():
    g = np.random.default_rng(7)
    K = g.normal(0, 1, (300, 8))
    q, w = g.normal(0, 1, (2, 8)), np.abs(g.normal(0, 1, 2))
    for t in (0, 3, 50, 401, 1199, 5000):
        sel = I.full_select(q, w, K, t, 64)
        assert all(4 * j + 3 <= t for j in sel["idx"])
        assert len(sel["idx"]) == min(64, I.n_visible(300, t))


def test_reuse_is_identity():
    idx = np.array([3, 9, 11, 400], dtype=np.int64)
    out = I.reuse_select(idx)
    assert np.array_equal(out, idx) and out is not idx
