"""Synthetic CSA2 workloads: shapes, seeds, length mixes, page tables and raw tensors.

Everything here is input *structure* and random data; none of the method's
arithmetic (compression, normalisation, rotation, quantisation, scoring,
selection, attention) lives in this module.  The CUDA path's tests and bench
and the CPU oracle both draw their inputs from here, so they see the same
numbers; each side then runs its own arithmetic on them.

Value recipe (same for every workload; each tensor has its own stream):
  hidden states          ~N(0,1), about 0.1% of elements replaced by +/-10, bf16
  projection weights     ~N(0, 0.02^2), bf16
  RMSNorm gain gamma     1 + 0.05*N(0,1), fp32
  cached latent (raw)    ~N(0,1), about 0.01% of channels replaced by +/-10, fp32
                         (each side normalises, rotates and packs it itself)
  indexer keys           ~N(0,1), bf16 (fp32 in the tiny workload)
  indexer queries        ~N(0,1), same dtype as the keys; head weights ~N(0,1) fp32
  attention queries Q    ~N(0,1), bf16
  sliding-window latent  ~N(0,1), fp32 (each side packs it to FP8 itself)
  replayed hidden states ~N(0,1), about 0.1% of elements replaced by +/-10, bf16, one
                         tensor per layer (window rebuilt by SWA Bounded Replay)
  page table             random permutation of the shared page pool
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

from . import rng

PAGE = 64  # compressed entries per KV page


@dataclass
class Workload:
    name: str
    seed: int
    B: int
    t_first: List[int]          # position of the first new token, per sequence
    n_new: int                  # new tokens per sequence this step (= query tokens)
    d: int = 512
    r: int = 64
    Hq: int = 64
    Hi: int = 8
    Di: int = 128
    K: int = 512
    W: int = 128
    idx_dtype: str = "bf16"     # "bf16" | "f32"
    H: Optional[int] = None     # hidden size when the step compresses its new tokens
    layers: List[str] = field(default_factory=lambda: ["F"])
    hierarchical: bool = False
    pool_blocks: int = 2048
    pool_block: int = 8
    rope_base: float = 10000.0
    eps: float = 1e-6
    replay_H: Optional[int] = None  # SWA Bounded Replay: hidden size of the replayed tokens
    kv_format: str = "mxfp4"    # main KV: "mxfp4" (the pages' V4.1 format) or "fp8" (V4-style, for the A/B)
    description: str = ""

    # ---- derived structure -------------------------------------------------
    @property
    def Tq(self) -> int:
        return self.n_new

    def entries_before(self, b: int) -> int:
        """Compressed entries already cached before this step (complete groups of 4).

        A replay step re-runs tokens whose compressed entries are already in the
        persistent cache: the cache then covers every replayed token too."""
        if self.replay_H is not None:
            return (self.t_first[b] + self.n_new) // 4
        return self.t_first[b] // 4

    def new_entries(self, b: int) -> int:
        """Entries this step produces (only when it compresses its new tokens)."""
        if self.H is None:
            return 0
        assert self.t_first[b] % 4 == 0, "a compressed chunk starts on a group boundary"
        return self.n_new // 4

    def entries_after(self, b: int) -> int:
        return self.entries_before(b) + self.new_entries(b)

    def q_pos(self) -> torch.Tensor:
        """int32 [B, Tq]: raw position of every query token."""
        t0 = torch.tensor(self.t_first, dtype=torch.int32).reshape(-1, 1)
        return t0 + torch.arange(self.n_new, dtype=torch.int32).reshape(1, -1)

    def pages_per_seq(self) -> List[int]:
        return [max(1, -(-self.entries_after(b) // PAGE)) for b in range(self.B)]

    @property
    def max_pages(self) -> int:
        return max(self.pages_per_seq())

    @property
    def n_pages(self) -> int:
        return sum(self.pages_per_seq())

    def page_table(self) -> torch.Tensor:
        """int32 [B, max_pages]: physical page of each logical page; -1 where unused."""
        perm = rng.permutation(rng.stream_key(self.seed, "pages"), self.n_pages)
        pt = torch.full((self.B, self.max_pages), -1, dtype=torch.int32)
        off = 0
        for b, n in enumerate(self.pages_per_seq()):
            pt[b, :n] = perm[off:off + n]
            off += n
        return pt

    # sliding-window rows held per sequence: the W-1 tokens before the first
    # new token (already packed state) plus the new tokens themselves; a replay
    # step rebuilds the window from its replayed tokens alone
    def swa_pos0(self) -> torch.Tensor:
        if self.replay_H is not None:
            return torch.tensor(self.t_first, dtype=torch.int32)
        return torch.tensor([max(0, t - (self.W - 1)) for t in self.t_first], dtype=torch.int32)

    @property
    def swa_cap(self) -> int:
        return self.n_new if self.replay_H is not None else (self.W - 1) + self.n_new

    def swa_rows_before(self, b: int) -> int:
        if self.replay_H is not None:
            return 0
        return self.t_first[b] - max(0, self.t_first[b] - (self.W - 1))

    # ---- raw tensors ---------------------------------------------------------
    def _key(self, *labels) -> int:
        return rng.stream_key(self.seed, *labels)

    def cache_latent(self, b: int, rows: torch.Tensor) -> torch.Tensor:
        """fp32 [len(rows), d]: raw latent of cached entries ``rows`` of sequence b."""
        rows = rows.to(torch.int64) + (b << 30)
        idx = rows.reshape(-1, 1) * self.d + torch.arange(
            self.d, dtype=torch.int64, device=rows.device).reshape(1, -1)
        v = rng.normal_at(self._key("cache_latent"), idx)
        return rng.with_outliers(self._key("cache_outlier"), idx, v, 10000, 10.0)

    def indexer_k(self, b: int, rows: torch.Tensor) -> torch.Tensor:
        """[len(rows), Di] indexer keys of cached entries ``rows`` of sequence b."""
        rows = rows.to(torch.int64) + (b << 30)
        v = rng.normal_rows(self._key("indexer_k"), self.Di, rows)
        return v.to(self.idx_torch_dtype)

    @property
    def idx_torch_dtype(self):
        return torch.bfloat16 if self.idx_dtype == "bf16" else torch.float32

    def idx_q(self, layer: int, device="cpu") -> torch.Tensor:
        v = rng.normal(self._key("idx_q", layer), (self.B, self.Tq, self.Hi, self.Di), device)
        return v.to(self.idx_torch_dtype)

    def idx_w(self, layer: int, device="cpu") -> torch.Tensor:
        return rng.normal(self._key("idx_w", layer), (self.B, self.Tq, self.Hi), device)

    def q(self, layer: int, device="cpu") -> torch.Tensor:
        v = rng.normal(self._key("q", layer), (self.B, self.Tq, self.Hq, self.d), device)
        return v.to(torch.bfloat16)

    # single query tokens (b, i) of the tensors above, element for element
    def idx_q_row(self, layer: int, b: int, i: int) -> torch.Tensor:
        n = self.Hi * self.Di
        v = rng.normal(self._key("idx_q", layer), (self.Hi, self.Di), offset=(b * self.Tq + i) * n)
        return v.to(self.idx_torch_dtype)

    def idx_w_row(self, layer: int, b: int, i: int) -> torch.Tensor:
        return rng.normal(self._key("idx_w", layer), (self.Hi,), offset=(b * self.Tq + i) * self.Hi)

    def q_row(self, layer: int, b: int, i: int) -> torch.Tensor:
        n = self.Hq * self.d
        v = rng.normal(self._key("q", layer), (self.Hq, self.d), offset=(b * self.Tq + i) * n)
        return v.to(torch.bfloat16)

    def swa_latent(self, layer: int, b: int, positions: torch.Tensor) -> torch.Tensor:
        """fp32 [len(positions), d]: raw sliding-window latent of raw tokens ``positions``."""
        return rng.normal_rows(self._key("swa", layer), self.d,
                               positions.to(torch.int64) + (b << 32))

    def hidden(self, device="cpu") -> torch.Tensor:
        """bf16 [B, n_new, H]: hidden states of the new tokens."""
        shape = (self.B, self.n_new, self.H)
        idx = torch.arange(self.B * self.n_new * self.H, dtype=torch.int64,
                           device=device).reshape(shape)
        v = rng.normal_at(self._key("hidden"), idx)
        v = rng.with_outliers(self._key("hidden_outlier"), idx, v, 1000, 10.0)
        return v.to(torch.bfloat16)

    def replay_hidden(self, layer: int, device="cpu") -> torch.Tensor:
        """bf16 [B, n_new, replay_H]: layer ``layer``'s hidden states of the replayed tokens."""
        shape = (self.B, self.n_new, self.replay_H)
        idx = torch.arange(self.B * self.n_new * self.replay_H, dtype=torch.int64, device=device).reshape(shape)
        return self._replay_values(layer, idx)

    def replay_hidden_rows(self, layer: int, b: int) -> torch.Tensor:
        """bf16 [n_new, replay_H]: sequence b of replay_hidden(layer), element for element."""
        n = self.n_new * self.replay_H
        idx = torch.arange(b * n, (b + 1) * n, dtype=torch.int64).reshape(self.n_new, self.replay_H)
        return self._replay_values(layer, idx)

    def _replay_values(self, layer: int, idx: torch.Tensor) -> torch.Tensor:
        v = rng.normal_at(self._key("replay_hidden", layer), idx)
        v = rng.with_outliers(self._key("replay_outlier", layer), idx, v, 1000, 10.0)
        return v.to(torch.bfloat16)

    def w_swa(self, layer: int, device="cpu") -> torch.Tensor:
        """bf16 [d, replay_H]: layer ``layer``'s projection of a token onto its window row."""
        return (rng.normal(self._key("w_swa", layer), (self.d, self.replay_H), device) * 0.02).to(torch.bfloat16)

    def w_compress(self, device="cpu") -> torch.Tensor:
        """bf16 [d, 4H]: the learned 4:1 compression map (row o = output channel o)."""
        return (rng.normal(self._key("w_c"), (self.d, 4 * self.H), device) * 0.02).to(torch.bfloat16)

    def w_index(self, device="cpu") -> torch.Tensor:
        """bf16 [Di, 4H]: projection of the concatenated group onto the indexer key."""
        return (rng.normal(self._key("w_i"), (self.Di, 4 * self.H), device) * 0.02).to(torch.bfloat16)

    def w_layers(self, n_layers: int, device="cpu") -> torch.Tensor:
        """bf16 [n_layers][d + Di][4H]: each layer's own compression map and indexer-key
        projection, stacked (the decoder layers' KV from one hidden state)."""
        out = torch.empty(n_layers, self.d + self.Di, 4 * self.H, dtype=torch.bfloat16, device=device)
        for l in range(n_layers):
            out[l] = (rng.normal(self._key("w_layer", l), (self.d + self.Di, 4 * self.H), device) * 0.02).to(
                torch.bfloat16)
        return out

    def gamma(self, device="cpu") -> torch.Tensor:
        return 1.0 + 0.05 * rng.normal(self._key("gamma"), (self.d,), device)

    def n_layers(self) -> int:
        return len(self.layers)


# ---- the five workloads ------------------------------------------------------

def _log_uniform_lengths(seed: int, n: int, lo: int, hi: int, label: str) -> List[int]:
    u = rng.uniform01(rng.stream_key(seed, label), n)
    return [int(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo)))) for x in u]


def tiny() -> Workload:
    """Tiny Full-mode layer: 256 tokens, hidden 256, d=64, indexer 4x32 fp32, K=16."""
    return Workload(name="tiny_full_t256", seed=0, B=1, t_first=[0], n_new=256, d=64, r=16,
                    Hq=4, Hi=4, Di=32, K=16, W=16, idx_dtype="f32", H=256,
                    description="1 sequence, 256-token prefill from position 0, "
                                "64 entries, d=64 (16 rope), Top-16, 4 heads, window 16")


def decode_128k(B: int = 32, L: int = 131072) -> Workload:
    """Decode, Full mode: B sequences, one new token after an L-token context."""
    return Workload(name=f"decode_full_{L // 1024}k_b{B}", seed=1, B=B, t_first=[L] * B, n_new=1,
                    description=f"{B} sequences x 1 new token at position {L}, "
                                f"{L // 4} entries each, Top-512, 64 heads, window 128")


def decode_fp8kv_128k(B: int = 32, L: int = 131072) -> Workload:
    """The decode workload with the V4-style FP8 main KV (E4M3 row + fp32 scale per
    entry, 516 B against MXFP4's 288 B): the A/B of the storage format."""
    wl = decode_128k(B, L)
    wl.kv_format = "fp8"
    wl.name = f"decode_fp8kv_{L // 1024}k_b{B}"
    wl.description += ", FP8 main KV (516 B/entry)"
    return wl


def prefill_64k(n_new: int = 4096, ctx: int = 65536, H: int = 4096) -> Workload:
    """Chunked prefill, Full mode: n_new tokens ending a ctx-token context, compressed 4:1."""
    return Workload(name=f"prefill_full_{ctx // 1024}k_chunk{n_new}", seed=2, B=1,
                    t_first=[ctx - n_new], n_new=n_new, H=H,
                    description=f"1 sequence, {n_new} new tokens at {ctx - n_new}..{ctx - 1}, "
                                f"hidden {H}, {ctx // 4} entries after the chunk")


def hierarchical_1m(B: int = 8, L: int = 1048576) -> Workload:
    """Decoder group at 1M context: Full + 3 Reindex + 3 Reuse layers, pooled indexer."""
    return Workload(name=f"hier_group_{L // 1024}k_b{B}", seed=3, B=B, t_first=[L] * B, n_new=1,
                    layers=["F", "X", "X", "X", "R", "R", "R"], hierarchical=True,
                    description=f"{B} sequences x 1 token at {L}, layers F,X,X,X,R,R,R, "
                                "pool 2048 blocks x 8")


def ragged_serving(B: int = 64, lo: int = 8192, hi: int = 1048576, n_short: int = 6) -> Workload:
    """Ragged paged decode batch, layers F + 5 Reuse.

    B - n_short sequences have contexts log-uniform in [lo, hi] tokens (at
    least 2,048 entries); n_short (about 10%) have contexts log-uniform in
    [64, 8188] tokens, i.e. fewer than 2,048 entries, so some fall below K
    entries and Top-K is truncated to the visible count.
    """
    long_ = _log_uniform_lengths(4, B - n_short, lo, hi, "ctx_long")
    short = _log_uniform_lengths(4, n_short, 64, 8188, "ctx_short")
    lengths = []
    si = 0
    li = 0
    for b in range(B):  # spread the short ones through the batch
        if n_short and b % (B // n_short) == 0 and si < n_short:
            lengths.append(short[si]); si += 1
        else:
            lengths.append(long_[li]); li += 1
    return Workload(name=f"ragged_paged_b{B}", seed=4, B=B, t_first=lengths, n_new=1,
                    layers=["F", "R", "R", "R", "R", "R"],
                    description=f"{B} sequences, contexts log-uniform {lo}..{hi} tokens "
                                f"plus {n_short} short ones log-uniform 64..8188, layers F + 5 R")


# ---- the pages' 40-layer mode schedule ("DeepSeek-V4.1 架构解析" §02) -------------------
# 18 encoder layers in three groups of six (one Full, five Reuse); 20 decoder
# layers in five groups (one Full + three Reuse, then four times one Reindex +
# three Reuse), the pool built by the decoder's Full layer.

ENCODER_LAYERS = (["F"] + ["R"] * 5) * 3
DECODER_LAYERS = ["F", "R", "R", "R"] + ["X", "R", "R", "R"] * 4


def encoder_stack(B: int = 32, L: int = 131072) -> Workload:
    """The 18 encoder layers' schedule on the decode shapes (one shared cache)."""
    return Workload(name=f"encoder_stack_{L // 1024}k_b{B}", seed=5, B=B, t_first=[L] * B, n_new=1,
                    layers=list(ENCODER_LAYERS),
                    description=f"{B} sequences x 1 token at {L}, 18 layers 3 x (F + 5 R)")


def decoder_stack(B: int = 32, L: int = 131072) -> Workload:
    """The 20 decoder layers' schedule on the decode shapes, pool from the Full layer."""
    return Workload(name=f"decoder_stack_{L // 1024}k_b{B}", seed=6, B=B, t_first=[L] * B, n_new=1,
                    layers=list(DECODER_LAYERS), hierarchical=True,
                    description=f"{B} sequences x 1 token at {L}, 20 layers (F + 3 R) + 4 x (X + 3 R), "
                                "pool 2048 blocks x 8")


def decoder_stack_prefill(n_new: int = 4096, ctx: int = 65536, H: int = 4096) -> Workload:
    """The decoder schedule on a prefill chunk: every query token's own pool, Reindex over it."""
    return Workload(name=f"decoder_stack_prefill_{ctx // 1024}k_chunk{n_new}", seed=7, B=1,
                    t_first=[ctx - n_new], n_new=n_new, H=H, layers=list(DECODER_LAYERS), hierarchical=True,
                    description=f"1 sequence, {n_new} new tokens at {ctx - n_new}..{ctx - 1}, hidden {H}, "
                                "20 layers (F + 3 R) + 4 x (X + 3 R), per-token pools")


def decoder_replay(B: int = 8, L: int = 131072, n_win: int = 128, H: int = 4096) -> Workload:
    """SWA Bounded Replay ("DeepSeek-V4.1 架构解析" §03) on the decoder: each of the 20
    decoder layers rebuilds its window from the last n_win tokens of every sequence
    and runs its step for those tokens, over the persistent compressed cache."""
    return Workload(name=f"decoder_replay_{L // 1024}k_b{B}_win{n_win}", seed=8, B=B, t_first=[L - n_win] * B,
                    n_new=n_win, layers=list(DECODER_LAYERS), hierarchical=True, replay_H=H,
                    description=f"{B} sequences, the last {n_win} of {L} tokens replayed through the 20 decoder "
                                f"layers (F + 3 R) + 4 x (X + 3 R): per layer window rows from hidden {H}, "
                                "then the layer step for the replayed tokens, per-token pools")


ALL = {
    "tiny": tiny,
    "decode": decode_128k,
    "decode_fp8kv": decode_fp8kv_128k,
    "prefill": prefill_64k,
    "hierarchical": hierarchical_1m,
    "ragged": ragged_serving,
    "encoder_stack": encoder_stack,
    "decoder_stack": decoder_stack,
    "decoder_stack_prefill": decoder_stack_prefill,
    "decoder_replay": decoder_replay,
}
