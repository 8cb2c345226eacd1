"""Counter-based seeded random numbers shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the attention method.  It only turns
(stream key, element counter) pairs into numbers, so that any slice of any
synthetic tensor can be regenerated on the host or on a GPU, bit for bit.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014).  The i-th output of a stream with key ``k``
is ``mix64(k + (i + 1) * GAMMA)`` with the published constants; for key 0
the first outputs are 0xe220a8397b1dcdaf, 0x6e789e6aa1b965f4, ...

Normal deviates: Irwin-Hall sum of twelve 16-bit uniforms (three SplitMix64
outputs per value), centred and scaled so the result has mean 0 and
variance 1 (up to 1/65536^2).  Only integer operations and one exact
int32 -> float32 conversion are used, so CPU and GPU produce identical
values: every value is an integer multiple of 2**-17 in [-6, 6].
"""
from __future__ import annotations

import torch

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB

_CHUNK = 1 << 22  # elements per generation chunk: bounds temporary memory


def _s64(u: int) -> int:
    """Two's-complement int64 value of an unsigned 64-bit constant."""
    u &= MASK64
    return u - (1 << 64) if u >= (1 << 63) else u


_GAMMA_S = _s64(GAMMA)
_MIX1_S = _s64(MIX1)
_MIX2_S = _s64(MIX2)


def _lsr(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 tensors holding unsigned 64-bit patterns."""
    return torch.bitwise_and(torch.bitwise_right_shift(x, s), (1 << (64 - s)) - 1)


def mix64(z: torch.Tensor) -> torch.Tensor:
    """SplitMix64 output function on int64 tensors (wrapping arithmetic)."""
    z = torch.bitwise_xor(z, _lsr(z, 30)) * _MIX1_S
    z = torch.bitwise_xor(z, _lsr(z, 27)) * _MIX2_S
    return torch.bitwise_xor(z, _lsr(z, 31))


def stream_key(seed: int, *labels) -> int:
    """Derive a 64-bit stream key from a seed and labels (str / int), on the host."""
    k = (seed * 0x2545F4914F6CDD1D + 0x1234567) & MASK64
    for lab in labels:
        if isinstance(lab, str):
            v = 0
            for ch in lab.encode():
                v = (v * 131 + ch) & MASK64
        else:
            v = int(lab) & MASK64
        k = _mix64_int((k ^ v) + GAMMA)
    return k


def _mix64_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def raw64(key: int, counters: torch.Tensor) -> torch.Tensor:
    """SplitMix64 outputs number ``counters`` (int64 tensor) of stream ``key``."""
    base = torch.full_like(counters, _s64(key))
    return mix64(base + (counters + 1) * _GAMMA_S)


def _normal_chunk(key: int, idx: torch.Tensor) -> torch.Tensor:
    acc = torch.zeros_like(idx)
    for j in range(3):
        z = raw64(key, idx * 3 + j)
        for s in (0, 16, 32, 48):
            acc = acc + torch.bitwise_and(_lsr(z, s) if s else z, 0xFFFF)
    # 2*sum - 12*65535 is an even integer in [-786420, 786420]: exact in float32
    v = (acc * 2 - 12 * 65535).to(torch.int32).to(torch.float32)
    return v * (1.0 / 131072.0)


def normal_at(key: int, idx: torch.Tensor) -> torch.Tensor:
    """Approximately N(0,1) float32 values for element counters ``idx`` (int64)."""
    flat = idx.reshape(-1)
    out = torch.empty(flat.shape, dtype=torch.float32, device=flat.device)
    for s in range(0, flat.numel(), _CHUNK):
        out[s:s + _CHUNK] = _normal_chunk(key, flat[s:s + _CHUNK])
    return out.reshape(idx.shape)


def uniform_bits_at(key: int, idx: torch.Tensor) -> torch.Tensor:
    """63 random bits (non-negative int64) per counter."""
    flat = idx.reshape(-1)
    out = torch.empty_like(flat)
    for s in range(0, flat.numel(), _CHUNK):
        out[s:s + _CHUNK] = _lsr(raw64(key, flat[s:s + _CHUNK]), 1)
    return out.reshape(idx.shape)


def normal(key: int, shape, device="cpu", offset: int = 0) -> torch.Tensor:
    """Tensor of the given shape; element with flat index i uses counter offset + i."""
    n = 1
    for s in shape:
        n *= int(s)
    idx = torch.arange(offset, offset + n, dtype=torch.int64, device=device)
    return normal_at(key, idx).reshape(tuple(shape))


def normal_rows(key: int, n_cols: int, rows: torch.Tensor) -> torch.Tensor:
    """Rows ``rows`` (int64 tensor) of a conceptual [*, n_cols] normal tensor."""
    idx = rows.to(torch.int64).reshape(-1, 1) * n_cols + torch.arange(
        n_cols, dtype=torch.int64, device=rows.device).reshape(1, -1)
    return normal_at(key, idx)


def with_outliers(key: int, idx: torch.Tensor, values: torch.Tensor, per: int,
                  magnitude: float) -> torch.Tensor:
    """Replace about one element in ``per`` by +/-magnitude (sign from a random bit)."""
    bits = uniform_bits_at(key, idx)
    hit = torch.remainder(torch.bitwise_right_shift(bits, 8), per) == 0
    sign = torch.where(torch.bitwise_and(bits, 1) == 1, -1.0, 1.0).to(values.dtype)
    return torch.where(hit, sign * magnitude, values)


def permutation(key: int, n: int) -> torch.Tensor:
    """A random permutation of range(n) (argsort of distinct random keys), on the host."""
    bits = uniform_bits_at(key, torch.arange(n, dtype=torch.int64))
    # a stable sort breaks the (practically impossible) ties by position
    order = torch.argsort(bits, stable=True)
    return order.to(torch.int32)


def uniform01(key: int, n: int) -> torch.Tensor:
    """float64 uniforms in [0, 1) with 53 random bits, on the host."""
    bits = uniform_bits_at(key, torch.arange(n, dtype=torch.int64))
    return torch.bitwise_right_shift(bits, 10).to(torch.float64) * (2.0 ** -53)
