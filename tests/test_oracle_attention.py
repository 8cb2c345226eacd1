"""Pins of oracle/attention.py and oracle/layer.py: closed forms, torch SDPA, dense masked form."""
import numpy as np
import torch

from csa2_inputs import workloads
from golden_io import load
from oracle import attention as A
from oracle import formats as F
from oracle import indexer as I
from oracle import layer as L

PAGE = load("page_constants.json")


def test_single_key_returns_its_value():
    g = np.random.default_rng(0)
    Q = g.normal(0, 1, (4, 16))
    k = g.normal(0, 1, (1, 16))
    O, lse = A.softmax_attention(Q, k, 0.25)
    assert np.allclose(O, np.repeat(k, 4, axis=0))
    assert np.allclose(lse, (Q @ k[0]) * 0.25)


def test_equal_logits_give_mean():
    g = np.random.default_rng(1)
    keys = g.normal(0, 1, (9, 8))
    O, lse = A.softmax_attention(np.zeros((3, 8)), keys, 1.0)
    assert np.allclose(O, keys.mean(axis=0)[None, :])
    assert np.allclose(lse, np.log(9))


def test_matches_torch_sdpa():
    g = torch.Generator().manual_seed(2)
    Q = torch.randn(8, 32, generator=g, dtype=torch.float64)
    Kk = torch.randn(50, 32, generator=g, dtype=torch.float64) * 2
    ref = torch.nn.functional.scaled_dot_product_attention(Q[None], Kk[None], Kk[None],
                                                           scale=1 / np.sqrt(32))[0]
    O, _ = A.softmax_attention(Q.numpy(), Kk.numpy(), 1 / np.sqrt(32))
    assert np.allclose(O, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_key_order_does_not_matter():
    g = np.random.default_rng(3)
    Q, keys = g.normal(0, 1, (2, 8)), g.normal(0, 1, (20, 8))
    p = g.permutation(20)
    assert np.allclose(A.softmax_attention(Q, keys, 0.3)[0], A.softmax_attention(Q, keys[p], 0.3)[0])


def test_window_positions():
    W = PAGE["swa_window"]["value"]
    assert list(A.window_positions(5, W)) == list(range(0, 6))
    w = A.window_positions(1000, W)
    assert len(w) == W and w[0] == 1000 - W + 1 and w[-1] == 1000


def test_all_visible_selection_equals_dense_causal_attention():
    """Top-K covering every visible entry reproduces dense masked causal attention."""
    g = np.random.default_rng(4)
    n, d, W, Hq = 40, 32, 16, 4
    kv = F.mxfp4_unpack(*F.mxfp4_pack(g.normal(0, 1, (n, d)).astype(np.float32)))
    swa_pos = np.arange(0, 200)
    swa = F.fp8_unpack_bf16(*F.fp8_pack(g.normal(0, 1, (200, d)).astype(np.float32)))
    Kidx = g.normal(0, 1, (n, 8))
    for t in (0, 2, 3, 50, 157, 199):
        Q = g.normal(0, 1, (Hq, d))
        sel = I.full_select(g.normal(0, 1, (2, 8)), np.ones(2), Kidx, t, k=n)["idx"]
        assert len(sel) == I.n_visible(n, t)
        win = A.window_positions(t, W)
        O, lse = A.sparse_attention(Q, kv[sel], swa[win], 1 / np.sqrt(d))
        Od, lsed = A.dense_causal_attention(Q, kv, t, swa, swa_pos, W, 1 / np.sqrt(d))
        assert np.allclose(O, Od, rtol=1e-10, atol=1e-12)
        assert np.allclose(lse, lsed, rtol=1e-12)


def test_tiny_layer_end_to_end_invariants():
    wl = workloads.tiny()
    samples = [(0, i) for i in range(0, 256, 5)] + [(0, 255)]
    out = L.run_group(wl, samples, want_scores=True)
    for (layer, b, i), r in out.items():
        t = r["t"]
        nv = I.n_visible(wl.entries_after(b), t)
        assert r["cnt"] == min(wl.K, nv)
        idx = r["idx"][:r["cnt"]]
        assert np.all(4 * idx + 3 <= t) and np.all(np.diff(idx) > 0)
        assert np.all(r["idx"][r["cnt"]:] == -1)
        assert len(r["scores"]) == nv
        assert np.all(np.isfinite(r["O"]))


def test_group_modes_reuse_and_reindex():
    wl = workloads.hierarchical_1m(B=2, L=4 * 20000)
    wl.Hq, wl.d, wl.r = 4, 64, 16   # keep the oracle quick; structure unchanged
    out = L.run_group(wl, [(1, 0)])
    full = out[(0, 1, 0)]
    assert len(full["pool"]) == PAGE["pool_blocks"]["value"]
    pos = I.pool_positions(full["pool"], 20000, 8)
    assert len(pos) == PAGE["pool_positions"]["value"]
    for layer in (1, 2, 3):                 # Reindex layers search only the pool
        r = out[(layer, 1, 0)]
        assert set(r["idx"][:r["cnt"]]).issubset(set(pos))
        assert r["cnt"] == 512
    assert np.array_equal(out[(4, 1, 0)]["idx"], out[(3, 1, 0)]["idx"])   # Reuse
    assert np.array_equal(out[(6, 1, 0)]["idx"], out[(3, 1, 0)]["idx"])
    assert not np.allclose(out[(4, 1, 0)]["O"], out[(5, 1, 0)]["O"])      # own Q per layer
