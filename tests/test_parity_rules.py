"""The comparison rules of parity.py for bytes packed after a GEMM, pinned on the CPU.

A "GPU" result is simulated with the oracle's own packers on values moved by
less than the error bound; the rules must accept it, and must reject the
mistakes a packing kernel could make: a scale off by one away from a rounding
boundary, a code two steps off, a one-step flip away from a boundary, a sign
flip away from zero, a bf16 key one step off away from a midpoint.
"""
import numpy as np
import pytest

import parity
from oracle import formats as F


def _rows(seed, n=64, d=512):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, d))
    x[rng.random((n, d)) < 1e-3] *= 8.0
    return (x / np.sqrt(np.mean(x * x, axis=1, keepdims=True))).astype(np.float32).astype(np.float64)


def _moved(x, tau, seed):
    """x moved by up to the bound (uniformly), rounded to fp32."""
    rng = np.random.default_rng(seed)
    return (x + tau * rng.uniform(-1.0, 1.0, x.shape)).astype(np.float32).astype(np.float64)


def test_mxfp4_rule_accepts_moves_within_the_bound():
    x = _rows(1)
    tau = np.full_like(x, 3e-4)
    for seed in range(4):
        codes, scales = F.mxfp4_pack(_moved(x, tau, seed).astype(np.float32))
        fs, fc = parity.check_mxfp4_after_gemm(codes, scales, x, tau)
        assert fc > 0 or seed > 0   # the move reaches some boundaries
    codes, scales = F.mxfp4_pack(x.astype(np.float32))
    assert parity.check_mxfp4_after_gemm(codes, scales, x, np.zeros_like(x)) == (0, 0)


def _first_group_away_from_boundaries(x):
    """Row, group and channel whose amax/6 and code decisions are far from every boundary."""
    for r in range(x.shape[0]):
        for g in range(x.shape[1] // 16):
            grp = x[r, 16 * g:16 * g + 16].astype(np.float32)
            u = float(np.float32(np.max(np.abs(grp)) / np.float32(6)))
            c = F.e4m3_encode(u)
            lo, hi = F.E4M3_TABLE[c - 1] if c else 0.0, F.E4M3_TABLE[c + 1]
            if abs(u - 0.5 * (F.E4M3_TABLE[c] + lo)) > 1e-2 * u and abs(u - 0.5 * (F.E4M3_TABLE[c] + hi)) > 1e-2 * u:
                s = F.E4M3_TABLE[c]
                v = np.abs(grp) / s
                mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
                far = np.min(np.abs(v[:, None] - mids[None, :]), axis=1) > 0.05
                ch = np.nonzero(far & (v > 0.8) & (v < 5.5))[0]
                if len(ch):
                    return r, g, 16 * g + int(ch[0])
    raise AssertionError("no group away from the boundaries")


def test_mxfp4_rule_rejects_packing_mistakes():
    x = _rows(2)
    tau = np.full_like(x, 1e-5)
    codes, scales = F.mxfp4_pack(x.astype(np.float32))
    r, g, ch = _first_group_away_from_boundaries(x)
    bad = scales.copy()
    bad[r, g] += 1                                 # a scale one code off, far from its boundary
    with pytest.raises(AssertionError):
        parity.check_mxfp4_after_gemm(codes, bad, x, tau)
    bad = scales.copy()
    bad[r, g] += 2                                 # two codes off
    with pytest.raises(AssertionError):
        parity.check_mxfp4_after_gemm(codes, bad, x, tau)
    byte, shift = ch // 2, 4 * (ch % 2)
    nib = (int(codes[r, byte]) >> shift) & 0xF
    for new in ((nib & 8) | ((nib & 7) + 1 if (nib & 7) < 7 else (nib & 7) - 1),   # one step, away from a boundary
                (nib & 8) | ((nib & 7) + 2 if (nib & 7) < 6 else (nib & 7) - 2),   # two steps
                nib ^ 8):                                                         # sign
        bad = codes.copy()
        bad[r, byte] = np.uint8((int(bad[r, byte]) & (0xFF ^ (0xF << shift))) | (new << shift))
        with pytest.raises(AssertionError):
            parity.check_mxfp4_after_gemm(bad, scales, x, tau)


def test_key_rule():
    rng = np.random.default_rng(3)
    k = rng.standard_normal(4096) * 2.0
    tau = np.full_like(k, 1e-4)
    # a move within the bound, rounded: accepted (small keys may move several steps)
    moved = _moved(k, tau, 4)
    stored = F.bf16_round(moved.astype(np.float32))
    assert parity.check_keys_after_gemm(stored, k, tau, "bf16") > 0
    ref = F.bf16_round(k.astype(np.float32))
    mids = np.abs(k - ref) / np.maximum(np.abs(ref), 1e-30)
    far = int(np.argmin(mids))        # the key closest to its bf16 value: far from a midpoint
    bad = ref.copy()
    bits = np.ascontiguousarray(np.array([bad[far]], np.float32)).view(np.uint32)
    bad[far] = float(((bits + (1 << 16)) & 0xFFFF0000).view(np.float32)[0])   # one bf16 step
    with pytest.raises(AssertionError):
        parity.check_keys_after_gemm(bad, k, tau, "bf16")
    with pytest.raises(AssertionError):
        parity.check_keys_after_gemm(k + 3 * tau, k, tau, "f32")
    assert parity.check_keys_after_gemm(k + 0.5 * tau, k, tau, "f32") == 0


def test_fp8_rule():
    x = _rows(5, n=32)
    tau = np.full_like(x, 2e-4)
    codes, scales = F.fp8_pack(_moved(x, tau, 6).astype(np.float32))
    parity.check_fp8_after_gemm(codes, scales, x, tau)
    codes, scales = F.fp8_pack(x.astype(np.float32))
    # a scale off by far more than the bound
    with pytest.raises(AssertionError):
        parity.check_fp8_after_gemm(codes, scales * np.float32(1.01), x, tau)
    # a code two steps off
    bad = codes.copy()
    i = int(np.argmax(np.abs(x[0])))
    bad[0, i] = (bad[0, i] & 0x80) | ((bad[0, i] & 0x7F) - 2)
    with pytest.raises(AssertionError):
        parity.check_fp8_after_gemm(bad, scales, x, tau)


def test_latent_bound_covers_a_perturbed_rmsnorm_rope():
    """The propagated bound covers what a perturbation of the GEMM output within its own
    bound does to the oracle's RMSNorm + RoPE rows."""
    from oracle import compress as Cm
    rng = np.random.default_rng(7)
    c = rng.standard_normal((16, 512)) * 2.5
    tau_c = np.abs(c) * 1e-4 + 1e-4
    gamma = 1.0 + 0.05 * rng.standard_normal(512)
    pos = 4 * np.arange(16) + 3
    x_ref = Cm.rope(Cm.rmsnorm(c, gamma, 1e-6), pos, 64, 10000.0)
    tau_x = parity.latent_error_bound(c, tau_c, gamma, 1e-6, 64, x_ref)
    for seed in range(8):
        c2 = c + tau_c * np.random.default_rng(seed).uniform(-1, 1, c.shape)
        x2 = Cm.rope(Cm.rmsnorm(c2, gamma, 1e-6), pos, 64, 10000.0)
        assert np.all(np.abs(x2 - x_ref) <= tau_x)
