"""End-to-end parity of the CUDA layer step with the oracle on seeded workloads.

Small workloads (several tiles, ragged tails) are checked on many query
tokens; the full-size workloads, in the launch configuration the bench times,
on sampled tokens.
"""
import math

import numpy as np
import pytest
import torch

import parity
from compressed_sparse_attention_05_gb300 import abi, build, harness
from csa2_inputs import workloads as WL
from oracle import attention as A
from oracle import indexer as I
from oracle import layer as OL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    abi.lib()


def _np(t):
    return t.detach().cpu().double().numpy()


def check_group(wl, samples, group=None):
    """Run the layer group on the GPU and compare sampled tokens with the oracle."""
    g = group or harness.LayerGroup(wl)
    g.step()
    torch.cuda.synchronize()
    assert abi.csa2_get_status() == 0
    tau = 1.0 / math.sqrt(wl.d)
    qpos = wl.q_pos()
    swaps = 0
    states = {}
    for (b, i) in samples:
        st = states.setdefault(b, OL.SequenceState(wl, b))
        t = int(qpos[b, i])
        Kall = st.indexer_keys()
        nv = I.n_visible(Kall.shape[0], t)
        prev = None
        pool = None
        for l, mode in enumerate(wl.layers):
            gi = g.idx[l][b, i].cpu().numpy()
            gc = int(g.cnt[l][b, i])
            if mode == "F":
                q, w = _np(wl.idx_q_row(l, b, i)), _np(wl.idx_w_row(l, b, i))
                s = I.index_scores(q, w, Kall[:nv])
                cond = I.score_condition(q, w, Kall[:nv])
                swaps += parity.check_topk_set(gi, gc, I.topk(s, wl.K), s, cond)
                if wl.hierarchical:
                    gp = g.pool[b, i].cpu().numpy()
                    gpc = int(g.pool_cnt[b, i])
                    bs = I.block_scores(s, 8)
                    bcond = np.array([cond[8 * k:8 * k + 8].max() for k in range(len(bs))])
                    swaps += parity.check_topk_set(gp, gpc, I.topk(bs, wl.pool_blocks), bs, bcond)
                    pool = gp[:gpc]
            elif mode == "X":
                q, w = _np(wl.idx_q_row(l, b, i)), _np(wl.idx_w_row(l, b, i))
                pos = I.pool_positions(pool, nv, 8)
                s = I.index_scores(q, w, Kall[pos])
                cond = I.score_condition(q, w, Kall[pos])
                ref = pos[I.topk(s, wl.K)]
                swaps += parity.check_topk_set(gi, gc, ref, s, cond, positions=pos)
            else:
                assert gc == prev[1] and np.array_equal(gi, prev[0])
            assert np.all(4 * gi[:gc] + 3 <= t), "causality"
            prev = (gi, gc)
            # attention with the GPU's (verified) selection
            Q = _np(wl.q_row(l, b, i))
            O, lse = A.sparse_attention(Q, st.kv_rows(gi[:gc]), st.swa_rows(l, OL.window_of(wl, b, t)), tau)
            err = parity.attn_err(g.O[l][b, i].cpu().numpy(), O)
            assert err <= parity.ATTN_RTOL, f"layer {l} ({mode}) token {(b, i)}: attention error {err}"
            # lse = log of the softmax normaliser; the kernels sum it from the fp32 or
            # the fp16-rounded weights (relative difference <= 2^-11 per weight)
            assert np.allclose(g.lse[l][b, i].cpu().numpy(), lse, rtol=0, atol=parity.LSE_ATOL)
    return g, swaps


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


def test_prefill_small_with_compression():
    wl = WL.prefill_64k(n_new=256, ctx=4096 + 256, H=256)
    g, _ = check_group(wl, [(0, i) for i in (0, 1, 2, 3, 4, 100, 254, 255)])
    # the new entries were packed by the fused compression epilogue: compare bytes
    st = OL.SequenceState(wl, 0)
    new = st.new_entries()
    ids = torch.from_numpy(new["entry_ids"])
    slots = g.page_table[0, ids // 64].long().cpu() * 64 + ids % 64
    codes = g.kv_codes[slots.cuda()].cpu().numpy()
    scales = g.kv_scales[slots.cuda()].cpu().numpy()
    # scales decided from the GEMM output: equal except at rounding boundaries
    assert (scales != new["scales"]).mean() < 0.01
    assert (codes != new["codes"]).mean() < 0.01
    kk = g.idx_k[slots.cuda()].float().cpu().double().numpy()
    assert np.allclose(kk, new["idx_k"], rtol=2e-2, atol=2e-2)


def test_prefill_batch2_with_compression():
    """Two sequences of 602 new tokens (150 entries each; the two trailing
    tokens make no entry): ragged 128-entry tiles and the batch stride of the
    compression GEMM, the many-rows Top-K, attention."""
    wl = WL.Workload(name="prefill_b2_small", seed=5, B=2, t_first=[4096, 2048], n_new=602, H=256,
                     description="2 sequences x 602 new tokens, hidden 256")
    g, _ = check_group(wl, [(0, 0), (0, 301), (0, 601), (1, 0), (1, 599), (1, 601)])
    for b in range(2):
        st = OL.SequenceState(wl, b)
        new = st.new_entries()
        assert len(new["entry_ids"]) == 150
        ids = torch.from_numpy(new["entry_ids"])
        slots = g.page_table[b, ids // 64].long().cpu() * 64 + ids % 64
        codes = g.kv_codes[slots.cuda()].cpu().numpy()
        scales = g.kv_scales[slots.cuda()].cpu().numpy()
        assert (scales != new["scales"]).mean() < 0.01
        assert (codes != new["codes"]).mean() < 0.01
        kk = g.idx_k[slots.cuda()].float().cpu().double().numpy()
        assert np.allclose(kk, new["idx_k"], rtol=2e-2, atol=2e-2)


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
    wl = WL.decode_128k()
    check_group(wl, [(0, 0), (31, 0)])


def test_full_hierarchical_1m_b8():
    wl = WL.hierarchical_1m()
    check_group(wl, [(5, 0)])


def test_full_ragged_b64():
    wl = WL.ragged_serving()
    lens = [wl.entries_before(b) for b in range(wl.B)]
    order = np.argsort(lens)
    check_group(wl, [(int(order[0]), 0), (int(order[5]), 0), (int(order[32]), 0)])


def test_full_prefill_64k():
    wl = WL.prefill_64k()
    check_group(wl, [(0, 0), (0, 2047), (0, 4095)])
