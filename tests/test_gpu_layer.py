"""End-to-end parity of the CUDA layer step with the oracle on seeded workloads.

Small workloads (several tiles, ragged tails) are checked on many query
tokens; the full-size workloads, in the launch configuration the bench times,
on sampled tokens.
"""
import numpy as np
import pytest
import torch

import parity
from compressed_sparse_attention_05_gb300 import abi, build, harness
from csa2_inputs import workloads as WL
from layer_check import _np, check_compressed_entries, check_group
from oracle import indexer as I
from oracle import layer as OL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    abi.lib()


def _decode_small():
    wl = WL.decode_128k(B=3, L=4096)
    wl.t_first = [20001, 4098, 777]
    wl.name = "decode_small"
    return wl


def test_tiny_full_layer():
    wl = WL.tiny()
    check_group(wl, [(0, i) for i in range(0, 256, 3)] + [(0, 255)])


def test_decode_small():
    wl = _decode_small()
    check_group(wl, [(0, 0), (1, 0), (2, 0)])


def test_decode_small_k1024():
    """Top-1024: nine 128-key chunks per token spread over a cluster of six CTAs
    (uneven head slices in the merge), a short last chunk on every rank."""
    wl = _decode_small()
    wl.K = 1024
    check_group(wl, [(0, 0), (1, 0), (2, 0)])


def test_decode_small_fp8kv():
    """The V4-style FP8 main KV: the packer writes E4M3 rows with fp32 scales and the
    attention kernel dequantises them as it does the window rows."""
    wl = _decode_small()
    wl.kv_format = "fp8"
    wl.name = "decode_small_fp8kv"
    g, _ = check_group(wl, [(0, 0), (1, 0), (2, 0)])
    assert g.kv_codes.shape[1] == wl.d and g.kv_scales.dtype == torch.float32


def test_prefill_small_with_compression_fp8kv():
    """Compression GEMM with the FP8 epilogue, then attention over FP8 entries."""
    wl = WL.prefill_64k(n_new=256, ctx=4096 + 256, H=256)
    wl.kv_format = "fp8"
    wl.name = "prefill_small_fp8kv"
    g, _ = check_group(wl, [(0, i) for i in (0, 1, 2, 3, 100, 255)])
    check_compressed_entries(g, wl, 0)


def test_decode_small_max_keys():
    """The largest key list the header admits: Top-2048 plus a 1,024-row window
    (24 chunks of 128 keys) spread over a cluster of 8 CTAs."""
    wl = _decode_small()
    wl.K, wl.W = 2048, 1024
    wl.name = "decode_small_max_keys"
    check_group(wl, [(0, 0), (1, 0), (2, 0)])


def test_prefill_small_max_keys():
    """One CTA per token over up to 17 chunks: every visible entry (Top-2048 of
    at most 1,088) plus a 1,024-row window."""
    wl = WL.prefill_64k(n_new=256, ctx=4096 + 256, H=256)
    wl.K, wl.W = 2048, 1024
    wl.name = "prefill_small_max_keys"
    check_group(wl, [(0, i) for i in (0, 1, 128, 255)])


@pytest.mark.parametrize("Hq", [128, 40])
def test_decode_small_head_groups(Hq):
    """Hq = 128: two groups of 64 heads (blockIdx.y), each merged over its own
    cluster; Hq = 40: one group with 24 zero-padded heads."""
    wl = _decode_small()
    wl.Hq = Hq
    wl.name = f"decode_small_hq{Hq}"
    check_group(wl, [(0, 0), (1, 0), (2, 0)])


def test_prefill_small_hq96():
    """One CTA per token (256 rows), 96 heads: a full group of 64 and a partial
    group of 32; every head's output and lse written by its own group only."""
    wl = WL.prefill_64k(n_new=256, ctx=4096 + 256, H=256)
    wl.Hq = 96
    wl.name = "prefill_small_hq96"
    g, _ = check_group(wl, [(0, i) for i in (0, 1, 100, 255)])
    assert torch.isfinite(g.lse[0]).all() and torch.isfinite(g.O[0]).all()   # every row and head written


def test_prefill_small_with_compression():
    wl = WL.prefill_64k(n_new=256, ctx=4096 + 256, H=256)
    g, _ = check_group(wl, [(0, i) for i in (0, 1, 2, 3, 4, 100, 254, 255)])
    check_compressed_entries(g, wl, 0)


def test_prefill_batch2_with_compression():
    """Two sequences of 602 new tokens (150 entries each; the two trailing
    tokens make no entry): ragged 128-entry tiles and the batch stride of the
    compression GEMM, the many-rows Top-K, attention."""
    wl = WL.Workload(name="prefill_b2_small", seed=5, B=2, t_first=[4096, 2048], n_new=602, H=256,
                     description="2 sequences x 602 new tokens, hidden 256")
    g, _ = check_group(wl, [(0, 0), (0, 301), (0, 601), (1, 0), (1, 599), (1, 601)])
    for b in range(2):
        assert len(OL.SequenceState(wl, b).new_entries()["entry_ids"]) == 150
        check_compressed_entries(g, wl, b)


def test_encoder_stack_small():
    """The pages' encoder schedule, 3 x (F + 5 R): three Full layers re-score
    the shared cache with their own queries; Reuse layers keep the indices."""
    wl = WL.encoder_stack(B=2, L=4 * 12000 + 1)
    check_group(wl, [(0, 0), (1, 0)])


def test_decoder_stack_small():
    """The pages' decoder schedule, (F + 3 R) + 4 x (X + 3 R), with the pool
    built by the Full layer and searched by every Reindex layer."""
    wl = WL.decoder_stack(B=2, L=4 * 20000 + 2)
    check_group(wl, [(0, 0), (1, 0)])


def test_decoder_stack_prefill_small():
    """The decoder schedule on a prefill chunk: each query token's own pool
    (block maxima from the indexer GEMM), Reindex over the per-token pools."""
    wl = WL.decoder_stack_prefill(n_new=96, ctx=4096 + 96, H=256)
    check_group(wl, [(0, 0), (0, 33), (0, 95)])


def test_decoder_replay_small():
    """SWA Bounded Replay on the decoder schedule: every layer rebuilds its window
    from its replayed tokens (csa2_swa_replay) and runs its step for them; the
    first replayed token sees only itself in the window, the last a full one."""
    wl = WL.decoder_replay(B=2, L=4 * 20000 + 40, n_win=40, H=256)
    check_group(wl, [(0, 0), (0, 39), (1, 17)])


def test_hierarchical_group_small():
    wl = WL.hierarchical_1m(B=2, L=4 * 20000 + 2)
    check_group(wl, [(0, 0), (1, 0)])


def test_ragged_small():
    wl = WL.ragged_serving(B=8, lo=2048, hi=120000, n_short=2)
    check_group(wl, [(b, 0) for b in range(8)])


def test_index_scores_tolerance():
    wl = _decode_small()
    g = harness.LayerGroup(wl)
    stride = g.max_entries
    scores = torch.full((wl.B, stride), float("nan"), device="cuda")
    bm = torch.full((wl.B, (stride + 7) // 8), float("nan"), device="cuda")
    abi.csa2_index_scores(g.dims(), g.cache(), g.idx_q[0], g.idx_w[0], g.q_pos, scores, bm)
    torch.cuda.synchronize()
    for b in range(wl.B):
        st = OL.SequenceState(wl, b)
        K = st.indexer_keys()
        t = wl.t_first[b]
        nv = I.n_visible(K.shape[0], t)
        q, w = _np(wl.idx_q_row(0, b, 0)), _np(wl.idx_w_row(0, b, 0))
        s_ref = I.index_scores(q, w, K[:nv])
        s_gpu = scores[b, :nv].cpu().numpy()
        assert parity.score_err(s_gpu, s_ref, I.score_condition(q, w, K[:nv])) <= parity.SCORE_RTOL
        # block maxima are exact maxima of the GPU's own scores
        ref_bm = I.block_scores(s_gpu, 8)
        assert np.array_equal(bm[b, :len(ref_bm)].cpu().double().numpy(), ref_bm)


def test_index_scores_many_queries():
    """Many query tokens per sequence (the tensor-core GEMM path): 80 tokens are
    two full 32-token blocks and a ragged one; every visible score of every
    token against the oracle on the keys as stored, block maxima exact."""
    wl = WL.prefill_64k(n_new=80, ctx=4096 + 80, H=256)
    g = harness.LayerGroup(wl)
    g.step()
    torch.cuda.synchronize()
    stride = g.max_entries
    rows = wl.B * wl.Tq
    scores = torch.full((rows, stride), float("nan"), device="cuda")
    bm = torch.full((rows, (stride + 7) // 8), float("nan"), device="cuda")
    abi.csa2_index_scores(g.dims(), g.cache(), g.idx_q[0], g.idx_w[0], g.q_pos, scores, bm)
    torch.cuda.synchronize()
    assert abi.csa2_get_status() == 0
    n_ent = wl.entries_after(0)
    ids = torch.arange(n_ent)
    slots = g.page_table[0, ids // 64].long().cpu() * 64 + ids % 64
    K = g.idx_k[slots.cuda()].float().cpu().double().numpy()
    qpos = wl.q_pos()
    for i in range(wl.Tq):
        nv = I.n_visible(n_ent, int(qpos[0, i]))
        q, w = _np(wl.idx_q_row(0, 0, i)), _np(wl.idx_w_row(0, 0, i))
        s_ref = I.index_scores(q, w, K[:nv])
        s_gpu = scores[i, :nv].cpu().numpy()
        assert parity.score_err(s_gpu, s_ref, I.score_condition(q, w, K[:nv])) <= parity.SCORE_RTOL, f"token {i}"
        ref_bm = I.block_scores(s_gpu, 8)
        assert np.array_equal(bm[i, :len(ref_bm)].cpu().double().numpy(), ref_bm), f"token {i}"


# ---- full-size workloads, sampled ------------------------------------------------------

def test_full_decode_128k_b32():
    """The bench's decode launch, 8 of its 32 tokens spread over the batch."""
    wl = WL.decode_128k()
    check_group(wl, [(b, 0) for b in (0, 3, 7, 12, 18, 24, 29, 31)])


def test_full_decode_fp8kv_128k_b32():
    wl = WL.decode_fp8kv_128k()
    check_group(wl, [(0, 0), (17, 0), (31, 0)])


def test_full_hierarchical_1m_b8():
    wl = WL.hierarchical_1m()
    check_group(wl, [(0, 0), (5, 0), (7, 0)])


def test_full_ragged_b64():
    wl = WL.ragged_serving()
    lens = [wl.entries_before(b) for b in range(wl.B)]
    order = np.argsort(lens)
    check_group(wl, [(int(order[0]), 0), (int(order[5]), 0), (int(order[32]), 0)])


def test_full_prefill_64k():
    """The 4,096-token chunk as the bench times it: every one of the 1,024 new
    entries (the 4H = 16,384 split-K compression GEMM over the [B][G][4H] tensor
    map) byte-checked, and 64 query tokens spread over all 128 blocks of 32
    tokens of the indexer GEMM and every lane position within a block."""
    wl = WL.prefill_64k()
    toks = sorted({0, wl.Tq - 1} | {32 * (2 * k + (k & 1)) + (5 * k) % 32 for k in range(63)})
    g, _ = check_group(wl, [(0, i) for i in toks])
    check_compressed_entries(g, wl, 0)
