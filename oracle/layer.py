"""One CSA2 layer step (or a group of layers) for sampled query tokens, in float64.

Test infrastructure only (see ``oracle/__init__.py``).

Composes the steps of ``compress``, ``formats``, ``indexer`` and ``attention``
in the order the pages give (DeepSeek-V4.1 architecture analysis
(blog.yuzhonghai.cloud), §02 and §03):

  Full     compress the new tokens (when the step has any), score every
           visible entry, Top-K; with the hierarchical indexer also the
           2,048-block pool; attend.
  Reindex  score only the pool of the most recent Full layer with this
           layer's own indexer query, Top-K, attend (KV and indexer K are
           the Full layer's).
  Reuse    take the previous layer's indices unchanged, attend.

Every layer has its own attention query Q and its own sliding window; the
compressed KV and the indexer keys are shared by the group.  A replay
workload (SWA Bounded Replay, §03) rebuilds each layer's window from its
replayed tokens (``replay``) and cuts the window at the first of them.

Inputs come from ``csa2_inputs.workloads`` (raw random tensors); every step
of arithmetic on them is done here.  The functions only touch the rows they
need, so single query tokens of the 1M-token workloads are affordable.
"""
from __future__ import annotations

import numpy as np
import torch

from . import attention, compress, formats, indexer, replay


def _np(x: torch.Tensor) -> np.ndarray:
    return x.detach().to("cpu").to(torch.float64).numpy()


class SequenceState:
    """Lazily built cache of one sequence: packed entries, indexer keys, window rows."""

    def __init__(self, wl, b: int):
        self.wl, self.b = wl, b
        self.n_before = wl.entries_before(b)
        self.n_after = wl.entries_after(b)
        self.gamma = _np(wl.gamma())
        self.kv_format = getattr(wl, "kv_format", "mxfp4")
        self._new = None
        self._idx_k = None
        self._replay = {}

    # new entries produced by this step's compression (Full layer of a prefill)
    def new_entries(self):
        if self._new is None and self.wl.H is not None:
            wl = self.wl
            hid = _np(wl.hidden()[self.b])
            self._new = compress.compress_pack(
                hid, _np(wl.w_compress()), self.gamma, wl.eps, wl.r, wl.rope_base,
                first_entry=self.n_before, W_idx=_np(wl.w_index()), idx_dtype=wl.idx_dtype,
                kv_format=self.kv_format)
        return self._new

    def indexer_keys(self) -> np.ndarray:
        """float64 [n_after, Di]: cached keys (synthetic) then the step's projected keys."""
        if self._idx_k is None:
            k = _np(self.wl.indexer_k(self.b, torch.arange(self.n_before)))
            new = self.new_entries()
            if new is not None:
                k = np.concatenate([k, new["idx_k"]], axis=0)
            self._idx_k = k
        return self._idx_k

    def packed_rows(self, rows: np.ndarray):
        """(codes, scales) of entries ``rows``: cached ones packed from the raw latent.

        MXFP4: codes [n, d/2], scales [n, d/16] (E4M3 codes); FP8 main KV: codes
        [n, d] (E4M3), scales [n] (fp32)."""
        rows = np.asarray(rows, dtype=np.int64)
        wl = self.wl
        fp8 = self.kv_format == "fp8"
        codes = np.zeros((len(rows), wl.d if fp8 else wl.d // 2), np.uint8)
        scales = np.zeros(len(rows), np.float32) if fp8 else np.zeros((len(rows), wl.d // 16), np.uint8)
        old = rows < self.n_before
        if old.any():
            lat = _np(wl.cache_latent(self.b, torch.from_numpy(rows[old])))
            pack = compress.norm_rope_pack_fp8 if fp8 else compress.norm_rope_pack
            _, c, s = pack(lat, rows[old], self.gamma, wl.eps, wl.r, wl.rope_base)
            codes[old], scales[old] = c, s
        if (~old).any():
            new = self.new_entries()
            k = rows[~old] - self.n_before
            codes[~old], scales[~old] = new["codes"][k], new["scales"][k]
        return codes, scales

    def kv_rows(self, rows) -> np.ndarray:
        c, s = self.packed_rows(rows)
        if self.kv_format == "fp8":
            return formats.fp8_unpack_bf16(c, s)
        return formats.mxfp4_unpack(c, s)

    def replay_rows(self, layer: int):
        """Window rows of layer ``layer`` rebuilt from the replayed tokens (SWA Bounded Replay)."""
        if layer not in self._replay:
            wl = self.wl
            self._replay[layer] = replay.window_rows(
                _np(wl.replay_hidden_rows(layer, self.b)), _np(wl.w_swa(layer)), self.gamma, wl.eps, wl.r,
                wl.rope_base, wl.t_first[self.b])
        return self._replay[layer]

    def swa_rows(self, layer: int, positions: np.ndarray) -> np.ndarray:
        """Dequantised window rows (bf16 values as float64) of raw tokens ``positions``."""
        positions = np.asarray(positions, dtype=np.int64)
        if self.wl.replay_H is not None:
            rows = self.replay_rows(layer)
            k = positions - self.wl.t_first[self.b]
            assert np.all((k >= 0) & (k < self.wl.n_new)), "the rebuilt window holds only replayed tokens"
            return formats.fp8_unpack_bf16(rows["codes"][k], rows["scales"][k])
        lat = _np(self.wl.swa_latent(layer, self.b, torch.from_numpy(positions)))
        codes, scales = formats.fp8_pack(lat)
        return formats.fp8_unpack_bf16(codes, scales)


def window_of(wl, b: int, t: int) -> np.ndarray:
    """Raw positions of the window rows the token at t of sequence b attends to: the
    last W tokens, cut at the first replayed token when the window was rebuilt."""
    if wl.replay_H is not None:
        return replay.replay_window_positions(t, wl.W, wl.t_first[b])
    return attention.window_positions(t, wl.W)


def run_group(wl, samples, layers=None, want_scores=False):
    """Run the workload's layer schedule for sampled query tokens.

    samples: list of (b, i) pairs (sequence, query token).  Returns a dict
    keyed by (layer, b, i) with idx (padded to K), cnt, O [Hq, d], lse [Hq],
    pool (Full hierarchical layers), and scores when want_scores.
    """
    layers = range(len(wl.layers)) if layers is None else layers
    qpos = wl.q_pos()
    tau = 1.0 / np.sqrt(wl.d)
    states = {}
    out = {}
    for (b, i) in samples:
        st = states.setdefault(b, SequenceState(wl, b))
        t = int(qpos[b, i])
        prev_idx = None
        pool = None
        for layer in range(len(wl.layers)):
            mode = wl.layers[layer]
            res = {}
            if mode == "F":
                q = _np(wl.idx_q_row(layer, b, i)); w = _np(wl.idx_w_row(layer, b, i))
                sel = indexer.full_select(q, w, st.indexer_keys(), t, wl.K, wl.hierarchical,
                                          wl.pool_blocks, wl.pool_block)
                idx = sel["idx"]
                if wl.hierarchical:
                    pool = sel["pool"]
                    res["pool"] = pool
                if want_scores:
                    res["scores"] = sel["scores"]
            elif mode == "X":
                assert pool is not None, "Reindex needs the pool of a preceding Full layer"
                q = _np(wl.idx_q_row(layer, b, i)); w = _np(wl.idx_w_row(layer, b, i))
                sel = indexer.reindex_select(q, w, st.indexer_keys(), t, wl.K, pool,
                                             wl.pool_block)
                idx = sel["idx"]
                if want_scores:
                    res["scores"] = sel["scores"]
                    res["positions"] = sel["positions"]
            elif mode == "R":
                idx = indexer.reuse_select(prev_idx)
            else:
                raise ValueError(mode)
            prev_idx = idx
            if layer in layers:
                Q = _np(wl.q_row(layer, b, i))
                swa_pos = window_of(wl, b, t)
                O, lse = attention.sparse_attention(Q, st.kv_rows(idx),
                                                    st.swa_rows(layer, swa_pos), tau)
                res.update(idx=indexer.pad(idx, wl.K), cnt=len(idx), O=O, lse=lse, t=t)
                out[(layer, b, i)] = res
    return out
