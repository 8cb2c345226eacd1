"""Pins of oracle/compress.py: closed forms, invariants, the pages' norm bound."""
import numpy as np
import torch

from golden_io import load
from oracle import compress as C
from oracle import formats as F

PAGE = load("page_constants.json")


def _hidden(T, H, seed=0):
    return np.random.default_rng(seed).normal(0, 1, (T, H))


def test_compression_ratio_and_partial_group():
    ratio = PAGE["compression_ratio"]["value"]
    h = _hidden(10, 3)
    W = np.random.default_rng(1).normal(0, 1, (5, ratio * 3))
    c = C.compress(h, W)
    assert c.shape == (10 // ratio, 5)       # the trailing 2 tokens make no entry


def test_selection_map_picks_token_and_channel():
    # W[o, k*H + h] = 1 selects channel h of token k of the group: c_j[o] = hidden[4j+k, h]
    T, H = 16, 6
    h = _hidden(T, H, 2)
    for k in range(4):
        for ch in (0, H - 1):
            W = np.zeros((1, 4 * H))
            W[0, k * H + ch] = 1.0
            c = C.compress(h, W)[:, 0]
            ref = h[np.arange(T // 4) * 4 + k, ch].astype(np.float32)
            assert np.array_equal(c, ref)


def test_averaging_map_gives_group_mean():
    T, H = 12, 4
    h = _hidden(T, H, 3)
    W = np.concatenate([np.eye(H)] * 4, axis=1) / 4.0
    c = C.compress(h, W)
    ref = h.reshape(T // 4, 4, H).mean(axis=1)
    assert np.allclose(c, ref, rtol=1e-6, atol=1e-7)


def test_compress_matches_torch_linear():
    T, H, d = 32, 8, 7
    h = _hidden(T, H, 4)
    W = np.random.default_rng(5).normal(0, 1, (d, 4 * H))
    ref = torch.nn.functional.linear(torch.from_numpy(h).reshape(T // 4, 4 * H),
                                     torch.from_numpy(W)).numpy()
    assert np.allclose(C.compress(h, W), ref.astype(np.float32), rtol=1e-6, atol=1e-6)


def test_rmsnorm_norm_is_sqrt_d_and_bounded():
    d = PAGE["latent_dim"]["value"]
    g = np.random.default_rng(6)
    c = g.normal(0, 3, (64, d))
    c[0, 5] = 1e4                                # a huge outlier channel
    x = C.rmsnorm(c, np.ones(d), 1e-6)
    assert np.allclose(np.linalg.norm(x, axis=1), np.sqrt(d), rtol=1e-6)
    bound = PAGE["latent_l2_bound"]
    assert abs(np.sqrt(d) - bound["value"]) < bound["tol"]
    assert np.abs(x).max() <= np.sqrt(d) + 1e-5  # |x_i| <= ||x|| = sqrt(d)


def test_rmsnorm_gain_and_scale_invariance():
    d = 64
    g = np.random.default_rng(7)
    c = g.normal(0, 1, (8, d))
    gamma = g.normal(1, 0.3, d)
    x1 = C.rmsnorm(c, np.ones(d), 1e-6)
    xg = C.rmsnorm(c, gamma, 1e-6)
    assert np.allclose(xg, x1 * gamma, rtol=2e-6, atol=1e-6)
    assert np.allclose(C.rmsnorm(c * 37.0, gamma, 1e-12), C.rmsnorm(c, gamma, 1e-12), rtol=2e-6)


def test_rope_is_complex_rotation_of_last_r_channels():
    d, r, base = 32, 8, 10000.0
    g = np.random.default_rng(8)
    x = g.normal(0, 1, (5, d))
    pos = np.array([0, 1, 7, 1000, 123457])
    y = C.rope(x, pos, r, base)
    assert np.array_equal(y[:, :d - r], x[:, :d - r].astype(np.float32))   # no-rope channels
    z = x[:, d - r:d - r // 2] + 1j * x[:, d - r // 2:]
    theta = base ** (-np.arange(r // 2) * 2.0 / r)
    zr = z * np.exp(1j * pos[:, None] * theta[None, :])
    assert np.allclose(y[:, d - r:d - r // 2], zr.real, atol=2e-6)
    assert np.allclose(y[:, d - r // 2:], zr.imag, atol=2e-6)
    assert np.array_equal(y[0], x[0].astype(np.float32))                     # position 0


def test_rope_norm_and_relative_position():
    d, r = 64, 16
    g = np.random.default_rng(9)
    x, y = g.normal(0, 1, (2, d))
    for p, q, s in [(3, 10, 5), (100, 7, 1000), (0, 0, 31)]:
        a = np.dot(C.rope(x[None], [p + s], r, 1e4)[0], C.rope(y[None], [q + s], r, 1e4)[0])
        b = np.dot(C.rope(x[None], [p], r, 1e4)[0], C.rope(y[None], [q], r, 1e4)[0])
        assert abs(a - b) < 1e-4
    xr = C.rope(x[None], [777], r, 1e4)[0]
    assert abs(np.linalg.norm(xr) - np.linalg.norm(x)) < 1e-5


def test_entry_position_is_last_token():
    assert list(C.entry_position([0, 1, 5])) == [3, 7, 23]


def test_compress_pack_pipeline_and_page_bounds():
    T, H, d, r = 64, 16, 512, 64
    g = np.random.default_rng(10)
    h = g.normal(0, 1, (T, H))
    W = g.normal(0, 0.3, (d, 4 * H))
    Wi = g.normal(0, 0.3, (32, 4 * H))
    gamma = np.ones(d)
    out = C.compress_pack(h, W, gamma, 1e-6, r, 1e4, first_entry=100, W_idx=Wi)
    x = C.rope(C.rmsnorm(C.compress(h, W), gamma, 1e-6), 4 * (100 + np.arange(T // 4)) + 3, r, 1e4)
    codes, scales = F.mxfp4_pack(x.astype(np.float32))
    assert np.array_equal(out["codes"], codes) and np.array_equal(out["scales"], scales)
    # after RMSNorm + RoPE the 512-d latent obeys the pages' bound; no group saturates
    assert np.abs(out["x"]).max() <= PAGE["latent_l2_bound"]["value"] + 0.05
    assert np.all(F.E4M3_TABLE[out["scales"]] * 6 < PAGE["mxfp4_max"]["value"])
    # indexer key projection: bf16 rounding of the same concatenation's product
    k = (C.concat_groups(h) @ Wi.T).astype(np.float32)
    assert np.array_equal(out["idx_k"], F.bf16_round(k))


def test_synthetic_latent_max_near_observed_value():
    from csa2_inputs import workloads
    wl = workloads.decode_128k(B=1, L=4096 * 16)
    lat = wl.cache_latent(0, torch.arange(4096)).double().numpy()
    x = C.rmsnorm(lat, np.ones(512), 1e-6)
    # the pages observe a largest magnitude around 10 after normalisation
    obs = PAGE["latent_observed_max"]["value"]
    assert 0.5 * obs < np.abs(x).max() < 2 * obs


def test_fp8_main_kv_pack_pipeline_and_error_bound():
    """V4-style FP8 main KV (kept for the A/B against MXFP4): the same RMSNorm + RoPE
    row, packed as E4M3 codes with one fp32 scale per entry (amax / 448)."""
    T, H, d, r = 64, 16, 512, 64
    g = np.random.default_rng(11)
    h = g.normal(0, 1, (T, H))
    W = g.normal(0, 0.3, (d, 4 * H))
    gamma = 1.0 + 0.1 * g.standard_normal(d)
    out = C.compress_pack(h, W, gamma, 1e-6, r, 1e4, first_entry=37, kv_format="fp8")
    mx = C.compress_pack(h, W, gamma, 1e-6, r, 1e4, first_entry=37)
    assert np.array_equal(out["x"], mx["x"])          # the format changes only the pack
    x = out["x"]
    assert out["codes"].shape == (T // 4, d) and out["scales"].dtype == np.float32
    # 516 bytes per entry (512 codes + one fp32 scale) against MXFP4's 288
    assert out["codes"][0].nbytes + out["scales"][:1].nbytes == 516
    assert mx["codes"][0].nbytes + mx["scales"][0].nbytes == PAGE["mxfp4_bytes_per_entry_d512"]["value"]
    # each row's largest magnitude lands on E4M3's largest finite value
    assert np.all(np.max(F.E4M3_TABLE[out["codes"] & 0x7F], axis=1) == PAGE["e4m3_max"]["value"])
    # error of one E4M3 rounding (3 mantissa bits: half a step is 2^-4 relative; below
    # the normal range half the 2^-9 subnormal step, scaled) then one bf16 rounding
    deq = F.fp8_unpack_bf16(out["codes"], out["scales"])
    s = out["scales"].astype(np.float64)[:, None]
    bound = (2.0 ** -4 * np.abs(x) + 2.0 ** -10 * s) * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(x)
    assert np.all(np.abs(deq - x) <= bound)
    # FP8 is the finer format: its error is well under MXFP4's on the same rows
    e8 = np.abs(deq - x).mean()
    e4 = np.abs(F.mxfp4_unpack(mx["codes"], mx["scales"]) - x).mean()
    assert e8 < 0.5 * e4
