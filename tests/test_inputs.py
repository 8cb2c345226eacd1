"""Pins for the shared seeded input generator (csa2_inputs)."""
import numpy as np
import torch

from csa2_inputs import rng, workloads

M64 = (1 << 64) - 1


def _splitmix_sequential(state, n):
    out = []
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_published_outputs():
    # published first outputs of SplitMix64 seeded with 0
    got = rng.raw64(0, torch.arange(3, dtype=torch.int64))
    got = [int(v) & M64 for v in got]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_form_matches_sequential_generator():
    key = rng.stream_key(7, "x", 3)
    got = [int(v) & M64 for v in rng.raw64(key, torch.arange(50, dtype=torch.int64))]
    assert got == _splitmix_sequential(key, 50)


def test_normal_is_exact_integer_form_and_standardised():
    key = rng.stream_key(1, "n")
    x = rng.normal(key, (200000,))
    assert x.dtype == torch.float32
    k = x.double() * 131072
    assert torch.all(k == torch.round(k))           # multiples of 2**-17
    assert float(x.abs().max()) <= 6.0
    assert abs(float(x.double().mean())) < 0.01
    assert abs(float(x.double().std()) - 1.0) < 0.01
    # independent recomputation of a few values from the sequential generator
    for i in (0, 1, 12345):
        zs = _splitmix_sequential(key, 3 * i + 3)[3 * i:3 * i + 3]
        s = sum((z >> sh) & 0xFFFF for z in zs for sh in (0, 16, 32, 48))
        assert float(x[i]) == (2 * s - 12 * 65535) / 131072.0


def test_slices_regenerate_identically():
    wl = workloads.decode_128k(B=4, L=4096)
    full = wl.q(0)
    assert torch.equal(wl.q_row(0, 2, 0), full[2, 0])
    qi = wl.idx_q(0)
    assert torch.equal(wl.idx_q_row(0, 3, 0), qi[3, 0])
    rows = torch.tensor([5, 1, 900])
    a = wl.cache_latent(1, rows)
    b = wl.cache_latent(1, torch.arange(1000))[rows]
    assert torch.equal(a, b)


def test_outlier_rate_and_page_table():
    wl = workloads.ragged_serving()
    pt = wl.page_table()
    used = pt[pt >= 0]
    assert used.numel() == wl.n_pages
    assert torch.equal(torch.sort(used).values, torch.arange(wl.n_pages, dtype=torch.int32))
    lat = wl.cache_latent(0, torch.arange(2000))
    frac = float((lat.abs() == 10.0).double().mean())
    assert 0.00003 < frac < 0.0003   # about 1 in 10,000 channels


def test_ragged_lengths_cover_truncation():
    wl = workloads.ragged_serving()
    n = [wl.entries_before(b) for b in range(wl.B)]
    assert sum(x < 2048 for x in n) == 6
    assert any(x < 512 for x in n)     # Top-512 truncates for some sequence
    assert max(n) <= 1048576 // 4


def test_replay_workload_layout():
    # SWA Bounded Replay: the queries are the last n_win tokens, the compressed
    # cache covers them, and each layer's window holds only the replayed rows
    wl = workloads.decoder_replay(B=3, L=4 * 3000 + 40, n_win=40, H=128)
    assert wl.Tq == 40 and wl.swa_cap == 40
    for b in range(wl.B):
        assert wl.entries_before(b) == wl.entries_after(b) == (4 * 3000 + 40) // 4
        assert wl.swa_rows_before(b) == 0
        assert int(wl.swa_pos0()[b]) == int(wl.q_pos()[b, 0]) == 4 * 3000
        assert torch.equal(wl.replay_hidden_rows(5, b), wl.replay_hidden(5)[b])
    assert not torch.equal(wl.replay_hidden(0), wl.replay_hidden(1))   # a stream per layer
    assert wl.w_swa(0).shape == (wl.d, 128) and not torch.equal(wl.w_swa(0), wl.w_swa(1))
