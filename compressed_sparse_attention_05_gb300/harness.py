"""Device state of one CSA2 layer group and the calls of one layer-group step.

Used by the tests and the bench to lay a synthetic workload out in HBM the way
include/csa2.h expects it, through the library's own kernels:

  KV page pool      kv_codes [n_pages*64, d/2] u8, kv_scales [n_pages*64, d/16] u8,
                    idx_k [n_pages*64, Di] (bf16 or fp32), one shared pool
  page table        [B, max_pages] int32 (random permutation of the pool)
  per layer         Q, indexer q / w, window buffers, outputs

Cached entries are written by csa2_norm_rope_pack from raw latent rows, window
rows by csa2_pack_swa_fp8 (or, for a replay workload, by csa2_swa_replay from
each layer's replayed hidden states inside the step), so no packing happens
outside the library.  The workload object (``wl``) supplies shapes and raw
random tensors only.
"""
from __future__ import annotations

import math
from typing import List, Optional

import torch

from . import abi

_CHUNK = 1 << 16  # cached entries packed per call while filling the pool


class LayerGroup:
    def __init__(self, wl, device: str = "cuda"):
        self.wl = wl
        self.device = device
        B, d, Di = wl.B, wl.d, wl.Di
        dev = torch.device(device)
        self.n_pages = wl.n_pages
        self.page_table = wl.page_table().to(dev)
        self.n_entries = torch.tensor([wl.entries_after(b) for b in range(B)], dtype=torch.int32, device=dev)
        self.max_entries = max(wl.entries_after(b) for b in range(B))
        n_slots = self.n_pages * 64
        self.fp8kv = getattr(wl, "kv_format", "mxfp4") == "fp8"
        if self.fp8kv:   # V4-style main KV: E4M3 row + fp32 scale per entry
            self.kv_codes = torch.zeros(n_slots, d, dtype=torch.uint8, device=dev)
            self.kv_scales = torch.zeros(n_slots, dtype=torch.float32, device=dev)
        else:
            self.kv_codes = torch.zeros(n_slots, d // 2, dtype=torch.uint8, device=dev)
            self.kv_scales = torch.zeros(n_slots, d // 16, dtype=torch.uint8, device=dev)
        self.idx_k = torch.zeros(n_slots, Di, dtype=wl.idx_torch_dtype, device=dev)
        self.gamma = wl.gamma(dev)
        self._fill_cache()

        self.q_pos = wl.q_pos().to(dev)
        self.first_entry = torch.tensor([wl.entries_before(b) for b in range(B)], dtype=torch.int32, device=dev)
        self.hidden = self.W_c = self.W_idx = None
        if wl.H is not None:
            self.hidden = wl.hidden(dev)
            self.W_c = wl.w_compress(dev)
            self.W_idx = wl.w_index(dev)

        L = len(wl.layers)
        rows = B * wl.Tq
        self.Q = [wl.q(l, dev) for l in range(L)]
        self.idx_q = [wl.idx_q(l, dev) if wl.layers[l] in "FX" else None for l in range(L)]
        self.idx_w = [wl.idx_w(l, dev) if wl.layers[l] in "FX" else None for l in range(L)]
        self.swa_pos0 = wl.swa_pos0().to(dev)
        self.replay = wl.replay_H is not None
        self.replay_hidden = self.W_swa = None
        if self.replay:   # SWA Bounded Replay: every layer's window rebuilt from its replayed tokens
            self.replay_hidden = [wl.replay_hidden(l, dev) for l in range(L)]
            self.W_swa = [wl.w_swa(l, dev) for l in range(L)]
            self.replay_pos0 = torch.tensor(wl.t_first, dtype=torch.int32, device=dev)
            self.replay_ws = torch.empty(max(256, abi.csa2_swa_replay_workspace_size(B, wl.n_new, wl.replay_H, d)),
                                         dtype=torch.uint8, device=dev)
        self.swa_codes, self.swa_scales, self.swa_new = [], [], []
        for l in range(L):
            codes = torch.zeros(B, wl.swa_cap, d, dtype=torch.uint8, device=dev)
            scales = torch.zeros(B, wl.swa_cap, dtype=torch.float32, device=dev)
            for b in range(B):
                n = wl.swa_rows_before(b)
                if n:
                    pos = torch.arange(wl.t_first[b] - n, wl.t_first[b], dtype=torch.int64, device=dev)
                    lat = wl.swa_latent(l, b, pos).contiguous()
                    abi.csa2_pack_swa_fp8(lat, codes[b, :n], scales[b, :n])
            self.swa_codes.append(codes)
            self.swa_scales.append(scales)
            if self.replay:
                self.swa_new.append(None)
                continue
            new = torch.stack([wl.swa_latent(l, b, self.q_pos[b].to(torch.int64)) for b in range(B)])
            self.swa_new.append(new.contiguous())

        # outputs; Reuse layers read and keep the previous layer's index buffers
        self.idx: List[torch.Tensor] = []
        self.cnt: List[torch.Tensor] = []
        for l in range(L):
            if wl.layers[l] == "R":
                self.idx.append(self.idx[-1])
                self.cnt.append(self.cnt[-1])
            else:
                self.idx.append(torch.full((B, wl.Tq, wl.K), -7, dtype=torch.int32, device=dev))
                self.cnt.append(torch.full((B, wl.Tq), -7, dtype=torch.int32, device=dev))
        self.pool = torch.full((B, wl.Tq, wl.pool_blocks), -7, dtype=torch.int32, device=dev)
        self.pool_cnt = torch.full((B, wl.Tq), -7, dtype=torch.int32, device=dev)
        self.O = [torch.full((B, wl.Tq, wl.Hq, d), float("nan"), dtype=torch.float32, device=dev) for _ in range(L)]
        self.lse = [torch.full((B, wl.Tq, wl.Hq), float("nan"), dtype=torch.float32, device=dev) for _ in range(L)]
        self.args = [self._layer_args(l) for l in range(L)]
        self._dims = self.dims()
        self._windows = [self.window(l) for l in range(L)]
        ws = max(abi.csa2_layer_workspace_size(a) for a in self.args)
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)

    # -- setup -------------------------------------------------------------------------
    def _fill_cache(self):
        wl = self.wl
        dev = self.kv_codes.device
        for b in range(wl.B):
            n = wl.entries_before(b)
            for s in range(0, n, _CHUNK):
                m = min(n, s + _CHUNK) - s
                rows = torch.arange(s, s + m, dtype=torch.int64, device=dev)
                lat = wl.cache_latent(b, rows).reshape(1, m, wl.d).contiguous()
                pack = abi.csa2_norm_rope_pack_fp8 if self.fp8kv else abi.csa2_norm_rope_pack
                pack(
                    lat, wl.r, self.gamma, wl.eps, wl.rope_base,
                    torch.tensor([s], dtype=torch.int32, device=dev),
                    torch.tensor([m], dtype=torch.int32, device=dev),
                    self.page_table[b:b + 1].contiguous(), self.n_pages, self.kv_codes, self.kv_scales)
                slots = self.page_table[b, rows // 64].to(torch.int64) * 64 + rows % 64
                self.idx_k[slots] = wl.indexer_k(b, rows)
        torch.cuda.synchronize(dev)

    def dims(self) -> abi.Dims:
        wl = self.wl
        return abi.Dims(B=wl.B, Tq=wl.Tq, d=wl.d, r=wl.r, Hq=wl.Hq, Hi=wl.Hi, Di=wl.Di,
                        idx_dtype=abi.CSA2_BF16 if wl.idx_dtype == "bf16" else abi.CSA2_F32, K=wl.K, W=wl.W,
                        max_pages=self.page_table.shape[1], n_pool_blocks=wl.pool_blocks,
                        pool_block=wl.pool_block, swa_cap=wl.swa_cap,
                        kv_format=abi.CSA2_KV_FP8 if self.fp8kv else abi.CSA2_KV_MXFP4)

    def cache(self) -> abi.Cache:
        return abi.Cache(kv_codes=self.kv_codes.data_ptr(), kv_scales=self.kv_scales.data_ptr(),
                         idx_k=self.idx_k.data_ptr(), page_table=self.page_table.data_ptr(),
                         n_entries=self.n_entries.data_ptr(), n_pages=self.n_pages)

    def window(self, layer: int) -> abi.Window:
        return abi.Window(codes=self.swa_codes[layer].data_ptr(), scales=self.swa_scales[layer].data_ptr(),
                          pos0=self.swa_pos0.data_ptr())

    def _layer_args(self, l: int) -> abi.LayerArgs:
        wl = self.wl
        mode = {"F": abi.MODE_FULL, "X": abi.MODE_REINDEX, "R": abi.MODE_REUSE}[wl.layers[l]]
        p = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
        a = abi.LayerArgs()
        a.mode = mode
        a.hierarchical = int(wl.hierarchical and mode == abi.MODE_FULL)
        a.dims = self.dims()
        a.cache = self.cache()
        a.window = self.window(l)
        a.q_pos = p(self.q_pos)
        a.max_entries = self.max_entries
        if mode == abi.MODE_FULL and self.hidden is not None:
            a.hidden, a.T, a.H = p(self.hidden), wl.n_new, wl.H
            a.W_c, a.W_idx = p(self.W_c), p(self.W_idx)
            a.first_entry = p(self.first_entry)
        a.gamma = p(self.gamma)
        a.eps, a.rope_base = wl.eps, wl.rope_base
        a.swa_new = p(self.swa_new[l])
        a.idx_q, a.idx_w = p(self.idx_q[l]), p(self.idx_w[l])
        a.Q = p(self.Q[l])
        a.softmax_scale = 1.0 / math.sqrt(wl.d)
        if mode == abi.MODE_REUSE:
            a.idx_in, a.cnt_in = p(self.idx[l - 1]), p(self.cnt[l - 1])
        a.idx_out, a.cnt_out = p(self.idx[l]), p(self.cnt[l])
        a.pool, a.pool_cnt = p(self.pool), p(self.pool_cnt)
        a.O, a.lse = p(self.O[l]), p(self.lse[l])
        return a

    # -- the step ------------------------------------------------------------------------
    def replay_window(self, l: int, stream=None):
        """Rebuild layer l's window from its replayed tokens (SWA Bounded Replay)."""
        wl = self.wl
        abi.csa2_swa_replay(self.replay_hidden[l], self.W_swa[l], self.gamma, wl.eps, wl.rope_base,
                            self.replay_pos0, self._dims, self._windows[l], self.replay_ws, stream)

    def step(self, layers: Optional[range] = None, stream=None):
        for l in (range(len(self.args)) if layers is None else layers):
            if self.replay:
                self.replay_window(l, stream)
            abi.csa2_layer(self.args[l], self.ws, stream)

    def step_inputs(self):
        """The per-step inputs a serving loop supplies (copied host->device in e2e runs)."""
        t = [*self.Q, *[x for x in self.idx_q if x is not None], *[x for x in self.idx_w if x is not None],
             *[x for x in self.swa_new if x is not None]]
        if self.hidden is not None:
            t.append(self.hidden)
        if self.replay:
            t.extend(self.replay_hidden)
        return t

    def step_outputs(self):
        return list(self.O)
