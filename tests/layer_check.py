"""Layer-group parity checks shared by the GPU tests and the smoke run.

check_group runs a workload's layer group through the C ABI and compares
sampled query tokens with the oracle (Top-K sets with near-threshold swaps,
pools, Reuse identity, causality, attention per token and head, lse);
check_compressed_entries compares the bytes this step's compression packed.
Rules and tolerances: parity.py.

Operands.  Each comparison runs the oracle on the same operands as the GPU
(the accuracy contract is stated "on the same dequantised operands"): the
selection is the GPU's (checked against the oracle's first), and so are the
packed KV rows and indexer keys, each verified byte for byte against the
oracle's own packing first -- equal, or a flip the boundary rule of parity.py
allows.  A legitimate flip moves one E2M1 code by one grid step (up to a third
of the value), so comparing attention against the oracle's own bytes would
charge the attention kernel for a packing decision already checked.
"""
import math

import numpy as np
import torch

import parity
from compressed_sparse_attention_05_gb300 import abi, harness
from oracle import attention as A
from oracle import compress as Cm
from oracle import formats as F
from oracle import indexer as I
from oracle import layer as OL


def _np(t):
    return t.detach().cpu().double().numpy()


class Operands:
    """The packed KV rows and indexer keys of sequence b as the GPU holds them, each
    verified against the oracle's packing before it is handed to the oracle."""

    def __init__(self, g, wl, b):
        self.g, self.wl, self.b = g, wl, b
        self.st = OL.SequenceState(wl, b)
        self.new = None
        if wl.H is not None:   # this step compressed new entries: verify them all once
            self.new = compressed_entry_bounds(wl, b)
            check_compressed_entries(g, wl, b)
        self._keys = None

    def slots(self, rows):
        rows = torch.as_tensor(np.asarray(rows, np.int64))
        return (self.g.page_table[self.b, rows // 64].long().cpu() * 64 + rows % 64).to(self.g.kv_codes.device)

    def indexer_keys(self):
        """float64 [n_after, Di]: cached keys (inputs, written by the harness) then the
        step's new keys as the GPU stored them (verified by check_compressed_entries)."""
        if self._keys is None:
            k = self.st.indexer_keys().copy()
            if self.new is not None:
                n0 = self.st.n_before
                ids = np.arange(n0, self.st.n_after)
                k[n0:] = self.g.idx_k[self.slots(ids)].float().cpu().double().numpy()
            self._keys = k
        return self._keys

    def kv_rows(self, rows):
        """Dequantised KV rows of entries ``rows`` from the GPU's bytes, after checking
        them against the oracle's packing (equal, or boundary flips)."""
        rows = np.asarray(rows, np.int64)
        sl = self.slots(rows)
        cg = self.g.kv_codes[sl].cpu().numpy()
        sg = self.g.kv_scales[sl].cpu().numpy()
        co, so = self.st.packed_rows(rows)
        fp8 = self.g.fp8kv
        diff = np.any(cg != co, axis=1) | (sg != so if fp8 else np.any(sg != so, axis=1))
        old = diff & (rows < self.st.n_before)
        if old.any():   # packed by csa2_norm_rope_pack(_fp8) from a given latent: fp32 rounding only
            wl = self.wl
            lat = _np(wl.cache_latent(self.b, torch.from_numpy(rows[old])))
            x, _, _ = Cm.norm_rope_pack(lat, rows[old], self.st.gamma, wl.eps, wl.r, wl.rope_base)
            tau = parity.latent_error_bound(lat, np.zeros_like(lat), self.st.gamma, wl.eps, wl.r, x)
            check = parity.check_fp8_after_gemm if fp8 else parity.check_mxfp4_after_gemm
            check(cg[old], sg[old], x, tau)
        assert not (diff & (rows >= self.st.n_before)).any() or self.new is not None
        return F.fp8_unpack_bf16(cg, sg) if fp8 else F.mxfp4_unpack(cg, sg)


def check_group(wl, samples, group=None):
    """Run the layer group on the GPU and compare sampled tokens with the oracle."""
    g = group or harness.LayerGroup(wl)
    g.step()
    torch.cuda.synchronize()
    assert abi.csa2_get_status() == 0
    tau = 1.0 / math.sqrt(wl.d)
    qpos = wl.q_pos()
    swaps = 0
    ops = {}
    for (b, i) in samples:
        op = ops.setdefault(b, Operands(g, wl, b))
        st = op.st
        t = int(qpos[b, i])
        Kall = op.indexer_keys()
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
            # attention with the GPU's (verified) selection and packed rows
            Q = _np(wl.q_row(l, b, i))
            O, lse = A.sparse_attention(Q, op.kv_rows(gi[:gc]), st.swa_rows(l, OL.window_of(wl, b, t)), tau)
            err = parity.attn_err(g.O[l][b, i].cpu().numpy(), O)
            assert err <= parity.ATTN_RTOL, f"layer {l} ({mode}) token {(b, i)}: attention error {err}"
            # lse = log of the softmax normaliser; the kernels sum it from the fp32 or
            # the fp16-rounded weights (relative difference <= 2^-11 per weight)
            assert np.allclose(g.lse[l][b, i].cpu().numpy(), lse, rtol=0, atol=parity.LSE_ATOL)
    return g, swaps


_BOUNDS = {}


def compressed_entry_bounds(wl, b):
    """(oracle post-RoPE rows x, their error bound tau_x, exact indexer keys, their bound)
    of the entries this step compresses for sequence b."""
    key = (wl.name, wl.seed, wl.B, wl.n_new, wl.H, tuple(wl.t_first), wl.kv_format, b)
    if key not in _BOUNDS:
        st = OL.SequenceState(wl, b)
        new = st.new_entries()
        cat = Cm.concat_groups(_np(wl.hidden()[b]))
        W, Wi = _np(wl.w_compress()), _np(wl.w_index())
        tau_x = parity.latent_error_bound(new["c"], parity.gemm_error_bound(cat, W), st.gamma, wl.eps, wl.r,
                                          new["x"])
        _BOUNDS[key] = (new, tau_x, cat @ Wi.T, parity.gemm_error_bound(cat, Wi))
    return _BOUNDS[key]


def check_compressed_entries(g, wl, b):
    """Entries packed by this step's compression (GEMM + RMSNorm/RoPE/MXFP4 or FP8
    epilogue) and their indexer keys, byte for byte against the oracle under the
    boundary rules of parity.check_mxfp4_after_gemm (check_fp8_after_gemm for the
    FP8 main KV) / check_keys_after_gemm.  Returns the flips."""
    new, tau_x, k_exact, tau_k = compressed_entry_bounds(wl, b)
    ids = torch.from_numpy(new["entry_ids"])
    slots = (g.page_table[b, ids // 64].long().cpu() * 64 + ids % 64).cuda()
    cg, sg = g.kv_codes[slots].cpu().numpy(), g.kv_scales[slots].cpu().numpy()
    if g.fp8kv:
        fs, fc = 0, parity.check_fp8_after_gemm(cg, sg, new["x"], tau_x)
    else:
        fs, fc = parity.check_mxfp4_after_gemm(cg, sg, new["x"], tau_x)
    fk = parity.check_keys_after_gemm(g.idx_k[slots].float().cpu().double().numpy(), k_exact, tau_k, wl.idx_dtype)
    return fs, fc, fk
