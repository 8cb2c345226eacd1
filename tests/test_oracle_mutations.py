"""Planted mistakes in the oracle (on the CPU) must make at least one pin fail.

Each case replaces one oracle function with a plausible wrong variant and
runs the pin that should catch it.
"""
import numpy as np
import pytest

import test_oracle_attention as TA
import test_oracle_compress as TC
import test_oracle_formats as TF
import test_oracle_indexer as TI
import test_oracle_replay as TR
from oracle import attention, compress, formats, indexer, replay


def _concat_feature_major(hidden):
    hidden = np.asarray(hidden, dtype=np.float64)
    T, H = hidden.shape
    return hidden[:T // 4 * 4].reshape(T // 4, 4, H).transpose(0, 2, 1).reshape(T // 4, 4 * H)


def _rms_no_gamma(c, gamma, eps):
    c = np.asarray(c, dtype=np.float64)
    return (c / np.sqrt(np.mean(c * c, axis=-1, keepdims=True) + eps)).astype(np.float32).astype(np.float64)


def _rms_sum(c, gamma, eps):
    c = np.asarray(c, dtype=np.float64)
    return (c / np.sqrt(np.sum(c * c, axis=-1, keepdims=True) + eps) * gamma).astype(np.float32).astype(np.float64)


_good_rope = compress.rope


def _rope_bad_sign(x, positions, r, base):
    return _good_rope(x, -np.asarray(positions, dtype=np.float64), r, base)


def _rope_adjacent_pairs(x, positions, r, base):
    x = np.array(x, dtype=np.float64)
    d = x.shape[-1]
    y = x.copy()
    perm = np.concatenate([np.arange(d - r), d - r + np.concatenate([np.arange(0, r, 2), np.arange(1, r, 2)])])
    y[:, perm] = x
    out = _good_rope(y, positions, r, base)
    return out[:, perm]


def _scores_no_relu(q, w, K):
    return ((np.asarray(K, np.float64) @ np.asarray(q, np.float64).T) @ np.asarray(w, np.float64)).astype(np.float32)


def _topk_ties_high(scores, k):
    s = np.asarray(scores, dtype=np.float64)
    n = s.shape[0]
    order = np.lexsort((-np.arange(n), -s))
    return np.sort(order[:min(k, n)])


def _n_visible_strict(n_entries, t):
    return int(max(0, min(n_entries, t // 4)))


def _block_sum(scores, block=8):
    s = np.asarray(scores, dtype=np.float64)
    n = s.shape[0]
    return np.array([np.sum(s[b * block:min(n, (b + 1) * block)]) for b in range(-(-n // block))])


def _attn_no_scale(Q, keys, tau):
    return _good_attn(Q, keys, 1.0)


_good_attn = attention.softmax_attention
_good_pack = formats.mxfp4_pack


def _pack_swapped_nibbles(x):
    c, s = _good_pack(x)
    return ((c >> 4) | ((c & 0xF) << 4)).astype(np.uint8), s


def _e4m3_ties_away(x):
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    mag = np.abs(x)
    best = np.zeros(x.shape, dtype=np.int64)
    best_d = np.full(x.shape, np.inf)
    for c, v in formats._E4M3_POS:
        dist = np.abs(v - mag)
        take = dist <= best_d       # ties go to the larger magnitude
        best = np.where(take, c, best)
        best_d = np.where(take, dist, best_d)
    return (best | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


_good_rows = replay.window_rows


def _rows_rotated_at_row_index(hidden, W_swa, gamma, eps, r, base, pos0):
    return _good_rows(hidden, W_swa, gamma, eps, r, base, 0)


def _rows_rotated_at_entry_position(hidden, W_swa, gamma, eps, r, base, pos0):
    return _good_rows(hidden, W_swa, gamma, eps, r, base, pos0 + 3)


def _replay_window_one_too_long(t, W, p0):
    return np.arange(max(p0, t - W), t + 1, dtype=np.int64)


def _replay_window_not_cut(t, W, p0):
    return np.arange(max(0, t - W + 1), t + 1, dtype=np.int64)


CASES = [
    ("compress", "concat_groups", _concat_feature_major, TC.test_selection_map_picks_token_and_channel),
    ("compress", "rmsnorm", _rms_no_gamma, TC.test_rmsnorm_gain_and_scale_invariance),
    ("compress", "rmsnorm", _rms_sum, TC.test_rmsnorm_norm_is_sqrt_d_and_bounded),
    ("compress", "rope", _rope_bad_sign, TC.test_rope_is_complex_rotation_of_last_r_channels),
    ("compress", "rope", _rope_adjacent_pairs, TC.test_rope_is_complex_rotation_of_last_r_channels),
    ("compress", "entry_position", lambda j: np.asarray(j, np.int64), TC.test_entry_position_is_last_token),
    ("indexer", "index_scores", _scores_no_relu, TI.test_scores_closed_forms),
    ("indexer", "topk", _topk_ties_high, TI.test_topk_all_equal_takes_lowest_indices_and_signed_zeros_tie),
    ("indexer", "n_visible", _n_visible_strict, TI.test_visibility_rule),
    ("indexer", "block_scores", _block_sum, TI.test_block_pool_by_entry_walk),
    ("attention", "softmax_attention", _attn_no_scale, TA.test_matches_torch_sdpa),
    ("formats", "mxfp4_pack", _pack_swapped_nibbles, TF.test_mxfp4_hand_example),
    ("formats", "e4m3_encode_array", _e4m3_ties_away, TF.test_e4m3_encoder_matches_torch_cast),
    ("replay", "window_rows", _rows_rotated_at_row_index, TR.test_window_row_is_compression_of_the_groups_last_token),
    ("replay", "window_rows", _rows_rotated_at_entry_position,
     TR.test_window_row_is_compression_of_the_groups_last_token),
    ("replay", "replay_window_positions", _replay_window_one_too_long,
     TR.test_replay_window_matches_brute_force_and_is_cut_at_the_replay_start),
    ("replay", "replay_window_positions", _replay_window_not_cut,
     TR.test_replay_window_matches_brute_force_and_is_cut_at_the_replay_start),
]

_MODULES = {"compress": compress, "indexer": indexer, "attention": attention, "formats": formats,
            "replay": replay}


@pytest.mark.parametrize("mod,name,bad,pin", CASES, ids=[f"{m}.{n}-{b.__name__}" for m, n, b, _ in CASES])
def test_planted_mistake_is_caught(monkeypatch, mod, name, bad, pin):
    monkeypatch.setattr(_MODULES[mod], name, bad)
    with pytest.raises(AssertionError):
        pin()
