"""The bench's algorithmic work per step (the numerators of its roofline
fractions), checked against figures derived by hand from the workload shapes.

Unit figures: 256 B of indexer key per visible entry (one 128-channel bf16
key, shared by the 8 indexer heads), 288 B per MXFP4 entry (256 B of E2M1
codes + 32 E4M3 scales for d = 512), 4 Hq d FLOP per (query, key) of attention
(QK^T and PV, 2 FLOP per multiply-add each), 2 Hi Di FLOP per (query, scored
entry) of the indexer."""
import bench
from csa2_inputs import workloads as WL

KEY_B = 128 * 2
ENTRY_B = 256 + 32


def test_decode_scan_and_gather_bytes():
    a = bench.algorithmic(WL.decode_128k())
    n = 131072 // 4                                      # entries per sequence
    assert a["scan_bytes"] == a["scan_bytes_per_launch"] == 32 * n * KEY_B == 268_435_456
    assert a["gathered_bytes"] == 32 * 512 * ENTRY_B
    assert a["pooled_bytes"] == 0
    # one token per sequence: 512 selected entries + 128 window rows per head
    assert a["attn_flops"] == 32 * (512 + 128) * 4 * 64 * 512


def test_hierarchical_bytes_per_sequence():
    a = bench.algorithmic(WL.hierarchical_1m())
    n = 1048576 // 4
    per_seq = n * KEY_B + 3 * 16384 * KEY_B + 7 * 512 * ENTRY_B   # F scan, 3 x pooled Reindex, 7 gathers
    assert per_seq == 80_723_968
    assert a["scan_bytes"] + a["pooled_bytes"] + a["gathered_bytes"] == 8 * per_seq
    assert a["scan_bytes_per_launch"] == 8 * n * KEY_B


def test_prefill_flops():
    wl = WL.prefill_64k()
    a = bench.algorithmic(wl)
    T, t0 = 4096, 65536 - 4096
    # every token of the chunk sees >= 15,360 entries and a full 128-token window
    assert a["attn_flops"] == a["attn_flops_per_launch"] == T * (512 + 128) * 4 * 64 * 512
    visible = sum(min(16384, (t0 + i + 1) // 4) for i in range(T))
    assert a["index_flops"] == 2 * visible * 8 * 128
    assert abs(a["index_flops"] / 1e9 - 133.1) < 0.05
    assert a["compress_flops"] == 2 * 1024 * (4 * 4096) * (512 + 128)


def test_replay_windows_start_at_the_first_replayed_token():
    wl = WL.decoder_replay(B=2, L=4 * 5000, n_win=40, H=256)
    a = bench.algorithmic(wl)
    per_token = [min(512, (wl.t_first[0] + i + 1) // 4) + min(128, i + 1) for i in range(40)]
    assert a["attn_flops"] == 2 * len(wl.layers) * sum(per_token) * 4 * wl.Hq * wl.d
    assert a["compress_flops"] == 2 * (2 * 40 * len(wl.layers)) * 256 * wl.d
