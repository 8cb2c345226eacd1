"""Number formats of the CSA2 KV cache, written out from their definitions.

Test infrastructure only (see ``oracle/__init__.py``).

Formats (DeepSeek-V4.1 architecture analysis (blog.yuzhonghai.cloud), §03
"precision and state rebuild"): the main KV is OCP MXFP4-style, E2M1 values
with one E4M3 scale per 16 channels and no second-level global scale; the
page quotes the largest representable magnitude as 448 x 6 = 2688.  The
sliding-window KV stays FP8 (E4M3), with one scale per token.

Every encoder here is "round to the nearest representable value, ties to the
value with the even code, magnitudes beyond the largest finite value clamp
to it (satfinite)", evaluated by brute force over all codes of the format.
Values that decide a code (x / scale) are formed in IEEE fp32, the
precision the CUDA kernels use, as the pages fix none.
"""
from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------
# bit-level decoders


def e2m1_decode_code(code: int) -> float:
    """Value of a 4-bit E2M1 code: 1 sign, 2 exponent (bias 1), 1 mantissa bit.

    Exponent field 0 is subnormal: value = m * 2**-1.  No inf / NaN codes.
    """
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = (m * 0.5) if e == 0 else (2.0 ** (e - 1)) * (1.0 + m * 0.5)
    return -mag if s else mag


def e4m3_decode_code(code: int) -> float:
    """Value of an 8-bit E4M3 (fn) code: 1 sign, 4 exponent (bias 7), 3 mantissa bits.

    Exponent field 0 is subnormal (m/8 * 2**-6); exponent 15 with mantissa 7
    is NaN; there is no infinity.  Largest finite magnitude 1.75 * 2**8 = 448.
    """
    s = (code >> 7) & 1
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return float("nan")
    mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


E2M1_TABLE = np.array([e2m1_decode_code(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_decode_code(c) for c in range(256)], dtype=np.float64)

# non-negative finite magnitudes with their codes (sign bit clear)
_E2M1_POS = [(c, E2M1_TABLE[c]) for c in range(8)]
_E4M3_POS = [(c, E4M3_TABLE[c]) for c in range(128) if not np.isnan(E4M3_TABLE[c])]


def _nearest_even_code(mag: float, candidates) -> int:
    """Code of the candidate nearest to mag; ties go to the even code.

    Magnitudes beyond the largest finite value saturate to it (satfinite):
    the clamp comes first, so the distances stay exact for huge inputs.
    """
    mag = min(mag, max(v for _, v in candidates))
    best_code, best_dist = None, None
    for c, v in candidates:
        dist = abs(v - mag)
        if best_dist is None or dist < best_dist or (dist == best_dist and c % 2 == 0):
            best_code, best_dist = c, dist
    return best_code


def e2m1_encode(x: float) -> int:
    """Round-to-nearest-even, satfinite E2M1 code of an fp32 value; the sign bit is kept."""
    x = float(np.float32(x))
    code = _nearest_even_code(abs(x), _E2M1_POS)
    return code | (8 if np.signbit(x) else 0)


def e4m3_encode(x: float) -> int:
    """Round-to-nearest-even, satfinite E4M3 code of an fp32 value; the sign bit is kept."""
    x = float(np.float32(x))
    code = _nearest_even_code(abs(x), _E4M3_POS)
    return code | (0x80 if np.signbit(x) else 0)


# vectorised forms (same rule, brute force over the candidate list) --------

def _encode_array(x: np.ndarray, candidates, sign_bit: int) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    # satfinite: clamp to the largest finite magnitude before measuring distances
    mag = np.minimum(np.abs(x), max(v for _, v in candidates))
    best = np.zeros(x.shape, dtype=np.int64)
    best_d = np.full(x.shape, np.inf)
    for c, v in candidates:
        dist = np.abs(v - mag)
        take = (dist < best_d) | ((dist == best_d) & (c % 2 == 0))
        best = np.where(take, c, best)
        best_d = np.where(take, dist, best_d)
    return (best | np.where(np.signbit(x), sign_bit, 0)).astype(np.uint8)


def e2m1_encode_array(x: np.ndarray) -> np.ndarray:
    return _encode_array(x, _E2M1_POS, 8)


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    return _encode_array(x, _E4M3_POS, 0x80)


# --------------------------------------------------------------------------
# bf16

def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even mantissa); returns float64.

    bf16 keeps the top 16 bits of the fp32 pattern.  Finite inputs only.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# MXFP4 main KV (a row of d channels = d/16 groups)

GROUP = 16


def mxfp4_pack_row(x: np.ndarray):
    """Pack one fp32 row into (codes uint8[d/2], scales uint8[d/16]).

    Per 16-channel group: scale code = E4M3(amax / 6) (fp32 division); if the
    scale decodes to 0 every code of the group is +0; otherwise each code is
    E2M1(x / scale) (fp32 division), so |dequantised| <= 6 * scale.  Two codes
    per byte, the even channel in the low nibble.
    """
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[0]
    assert d % GROUP == 0
    codes4 = np.zeros(d, dtype=np.uint8)
    scales = np.zeros(d // GROUP, dtype=np.uint8)
    for g in range(d // GROUP):
        grp = x[g * GROUP:(g + 1) * GROUP]
        amax = np.float32(np.max(np.abs(grp)))
        sc = e4m3_encode(np.float32(amax / np.float32(6.0)))
        scales[g] = sc
        s = np.float32(E4M3_TABLE[sc])
        if s == 0:
            continue
        q = (grp / s).astype(np.float32)
        codes4[g * GROUP:(g + 1) * GROUP] = e2m1_encode_array(q)
    packed = (codes4[0::2] | (codes4[1::2] << 4)).astype(np.uint8)
    return packed, scales


def mxfp4_pack(x: np.ndarray):
    """Row-wise MXFP4 pack of an [n, d] fp32 array -> (codes [n, d/2], scales [n, d/16])."""
    x = np.asarray(x, dtype=np.float32)
    n, d = x.shape
    codes = np.zeros((n, d // 2), dtype=np.uint8)
    scales = np.zeros((n, d // GROUP), dtype=np.uint8)
    if n == 0:
        return codes, scales
    # same rule as mxfp4_pack_row, vectorised over rows and groups
    g = x.reshape(n, d // GROUP, GROUP)
    amax = np.max(np.abs(g), axis=2).astype(np.float32)
    sc = e4m3_encode_array((amax / np.float32(6.0)).astype(np.float32))
    s = E4M3_TABLE[sc].astype(np.float32)
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    q = (g / safe[:, :, None]).astype(np.float32)
    c4 = e2m1_encode_array(q)
    c4 = np.where((s == 0)[:, :, None], 0, c4).astype(np.uint8).reshape(n, d)
    codes[:] = c4[:, 0::2] | (c4[:, 1::2] << 4)
    scales[:] = sc
    return codes, scales


def mxfp4_unpack(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantise [n, d/2] codes and [n, d/16] scales to float64 [n, d] (exact)."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    n, half = codes.shape
    d = half * 2
    c4 = np.empty((n, d), dtype=np.uint8)
    c4[:, 0::2] = codes & 0xF
    c4[:, 1::2] = codes >> 4
    vals = E2M1_TABLE[c4]
    s = E4M3_TABLE[scales]
    return vals * np.repeat(s, GROUP, axis=1)


# --------------------------------------------------------------------------
# FP8 sliding-window KV (one fp32 scale per token row)

def fp8_pack(x: np.ndarray):
    """Pack [n, d] fp32 rows -> (codes uint8 [n, d], scales fp32 [n]).

    scale = amax / 448 (fp32 division, stored as fp32); scale 0 gives all-zero
    codes; codes = E4M3(x / scale) (fp32 division, satfinite).
    """
    x = np.asarray(x, dtype=np.float32)
    n, d = x.shape
    amax = np.max(np.abs(x), axis=1).astype(np.float32) if n else np.zeros(0, np.float32)
    s = (amax / np.float32(448.0)).astype(np.float32)
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    q = (x / safe[:, None]).astype(np.float32)
    codes = e4m3_encode_array(q)
    codes = np.where((s == 0)[:, None], 0, codes).astype(np.uint8)
    return codes, s


def fp8_unpack_bf16(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantise to the attention operand: bf16( fp32( e4m3(code) * scale ) ), as float64."""
    v = E4M3_TABLE[np.asarray(codes, dtype=np.uint8)].astype(np.float32)
    prod = (v * np.asarray(scales, dtype=np.float32)[:, None]).astype(np.float32)
    return bf16_round(prod)
