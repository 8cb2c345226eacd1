"""Pins of oracle/replay.py (SWA Bounded Replay): a reduction to the compression
pipeline, a library routine, the norm invariant and brute-force window sets."""
import numpy as np
import torch

from golden_io import load
from oracle import attention as A
from oracle import compress as C
from oracle import formats as F
from oracle import replay as R

PAGE = load("page_constants.json")


def _rng(seed):
    return np.random.default_rng(seed)


def test_window_row_is_compression_of_the_groups_last_token():
    # W = [0, 0, 0, W_swa] makes entry j of the compression the projection of
    # token 4j+3, rotated at 4j+3: the window row of that token, at its own raw
    # position, is the same latent (the compression itself is pinned elsewhere)
    n, H, d, r, base, eps = 24, 16, 64, 16, 10000.0, 1e-6
    pos0 = 4 * 10                                   # replay starts on a group boundary, not at 0
    g = _rng(1)
    hidden = g.normal(0, 1, (n, H))
    W_swa = g.normal(0, 0.3, (d, H))
    gamma = 1.0 + 0.05 * g.normal(0, 1, d)
    W4 = np.concatenate([np.zeros((d, 3 * H)), W_swa], axis=1)
    ref = C.compress_pack(hidden, W4, gamma, eps, r, base, first_entry=pos0 // 4)
    rows = R.window_rows(hidden, W_swa, gamma, eps, r, base, pos0)
    assert rows["x"].shape == (n, d) and rows["codes"].shape == (n, d) and rows["scales"].shape == (n,)
    np.testing.assert_allclose(rows["x"][3::4], ref["x"], rtol=1e-6, atol=1e-6)
    codes, scales = F.fp8_pack(ref["x"].astype(np.float32))
    assert np.array_equal(rows["codes"][3::4], codes)
    assert np.array_equal(rows["scales"][3::4], scales)


def test_projection_matches_torch_linear():
    g = _rng(2)
    hidden = g.normal(0, 1, (9, 32))
    W = g.normal(0, 1, (7, 32))
    ref = torch.nn.functional.linear(torch.from_numpy(hidden), torch.from_numpy(W)).numpy()
    np.testing.assert_allclose(R.project(hidden, W), ref.astype(np.float32), rtol=1e-6, atol=1e-6)


def test_rows_have_the_rmsnorm_norm_and_fp8_range():
    d = PAGE["latent_dim"]["value"]
    g = _rng(3)
    hidden = g.normal(0, 1, (12, 64))
    hidden[3, 7] = 50.0                              # an outlier token
    rows = R.window_rows(hidden, g.normal(0, 0.1, (d, 64)), np.ones(d), 1e-6, 64, 10000.0, pos0=1001)
    # unit gain: every row has L2 norm sqrt(d) after RMSNorm, and RoPE keeps it
    np.testing.assert_allclose(np.linalg.norm(rows["x"], axis=1), np.sqrt(d), rtol=1e-5)
    deq = F.E4M3_TABLE[rows["codes"]] * rows["scales"][:, None]
    assert np.all(np.abs(deq) <= PAGE["e4m3_max"]["value"] * rows["scales"][:, None] * (1 + 1e-7))
    # the row's largest magnitude lands on the largest E4M3 value
    top = np.argmax(np.abs(rows["x"]), axis=1)
    assert np.all(np.abs(F.E4M3_TABLE[rows["codes"][np.arange(12), top]]) == PAGE["e4m3_max"]["value"])


def test_replay_window_matches_brute_force_and_is_cut_at_the_replay_start():
    n_win = PAGE["swa_window"]["value"]
    for p0 in (0, 5, 1000):
        for W in (1, 4, n_win):
            for t in range(p0, p0 + 3 * n_win, 7):
                brute = [q for q in range(t + 1) if q >= p0 and t - q < W]
                assert list(R.replay_window_positions(t, W, p0)) == brute
            # the first replayed token sees only itself; from p0 + W - 1 on the window is full
            assert list(R.replay_window_positions(p0, W, p0)) == [p0]
            assert len(R.replay_window_positions(p0 + W - 1, W, p0)) == W
    # a replay that starts at the sequence start is the exact window
    for t in (0, 3, 127, 128, 5000):
        assert np.array_equal(R.replay_window_positions(t, n_win, 0), A.window_positions(t, n_win))
