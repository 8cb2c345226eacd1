"""Pins of oracle/formats.py: published format definitions, page constants, library casts."""
import numpy as np
import pytest
import torch

from golden_io import load
from oracle import formats as F

PAGE = load("page_constants.json")
OCP = load("ocp_formats.json")


def test_e2m1_decoder_matches_published_values():
    pos = [F.E2M1_TABLE[c] for c in range(8)]
    assert pos == OCP["e2m1_positive_values"]
    neg = [F.E2M1_TABLE[c] for c in range(8, 16)]
    assert neg == [-v for v in OCP["e2m1_positive_values"]]
    assert np.signbit(F.E2M1_TABLE[8])        # code 0x8 is -0


def test_e4m3_decoder_matches_published_values():
    for code, val in OCP["e4m3_examples"].items():
        assert F.E4M3_TABLE[int(code, 16)] == val
    finite = F.E4M3_TABLE[~np.isnan(F.E4M3_TABLE)]
    assert finite.max() == OCP["e4m3_max_normal"]
    assert np.min(np.abs(finite[finite != 0])) == OCP["e4m3_min_subnormal"]
    assert [c for c in range(256) if np.isnan(F.E4M3_TABLE[c])] == OCP["e4m3_nan_codes"]
    assert not np.isinf(F.E4M3_TABLE).any()


def test_page_range_constant():
    # largest MXFP4 magnitude = largest E2M1 value x largest E4M3 scale
    assert F.E2M1_TABLE.max() == PAGE["e2m1_max"]["value"]
    assert np.nanmax(F.E4M3_TABLE) == PAGE["e4m3_max"]["value"]
    assert F.E2M1_TABLE.max() * np.nanmax(F.E4M3_TABLE) == PAGE["mxfp4_max"]["value"]
    codes, scales = F.mxfp4_pack(np.full((1, 16), 1e9, np.float32))
    assert F.mxfp4_unpack(codes, scales).max() == PAGE["mxfp4_max"]["value"]


def test_e4m3_encoder_matches_torch_cast():
    g = torch.Generator().manual_seed(0)
    x = torch.cat([torch.randn(20000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x.clamp(-448, 448)
    # exact ties between neighbouring E4M3 values
    mids = []
    for c in range(1, 126):
        a, b = F.E4M3_TABLE[c], F.E4M3_TABLE[c + 1]
        mids += [(a + b) / 2, -(a + b) / 2]
    x = torch.cat([x, torch.tensor(mids, dtype=torch.float32)])
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.e4m3_encode_array(x.numpy())
    assert np.array_equal(got, ref)


def test_e4m3_saturates():
    assert F.e4m3_encode(500.0) == 0x7E
    assert F.e4m3_encode(-1e30) == 0xFE
    assert F.e4m3_encode(3e38) == 0x7E
    assert np.array_equal(F.e4m3_encode_array(np.array([1e38, -2e37], np.float32)), [0x7E, 0xFE])
    assert np.array_equal(F.e2m1_encode_array(np.array([1e38, -2e37], np.float32)), [0x7, 0xF])
    assert F.e4m3_encode(0.0) == 0x00
    assert F.e4m3_encode(-0.0) == 0x80


@pytest.mark.parametrize("x,code", [
    (0.25, 0x0), (0.26, 0x1), (0.75, 0x2), (1.25, 0x2), (1.26, 0x3), (1.75, 0x4),
    (2.5, 0x4), (2.6, 0x5), (3.5, 0x6), (5.0, 0x6), (5.1, 0x7), (7.0, 0x7), (1e9, 0x7),
    (-0.1, 0x8), (-1.75, 0xC), (-6.0, 0xF), (0.5, 0x1), (3.0, 0x5),
    (2.2e35, 0x7), (-3e38, 0xF),
])
def test_e2m1_round_to_nearest_even(x, code):
    assert F.e2m1_encode(x) == code


def test_e2m1_nearest_value_brute_force():
    g = np.random.default_rng(1)
    x = np.concatenate([g.normal(0, 3, 5000), g.uniform(-7, 7, 5000)]).astype(np.float32)
    codes = F.e2m1_encode_array(x)
    v = F.E2M1_TABLE[codes]
    grid = np.unique(np.abs(F.E2M1_TABLE))
    best = np.min(np.abs(np.abs(x)[:, None] - grid[None, :]), axis=1)
    assert np.allclose(np.abs(np.abs(x) - np.abs(v)), best, atol=0)
    assert np.all((np.sign(v) == np.sign(x)) | (v == 0))


def test_bf16_round_matches_torch():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(100000, generator=g) * 100
    # exact ties: pattern with the lower 16 bits 0x8000
    u = (torch.randint(0, 1 << 15, (1000,), generator=g, dtype=torch.int32) << 16) | 0x8000
    x = torch.cat([x, u.view(torch.float32)])
    x = x[torch.isfinite(x)]
    ref = x.to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.bf16_round(x.numpy()), ref)


def test_mxfp4_hand_example():
    row = np.zeros(32, np.float32)
    row[:5] = [6.0, -3.0, 1.25, 0.1, 2.5]
    row[16:18] = [0.0, -0.0]                     # an all-zero group
    codes, scales = F.mxfp4_pack(row[None, :])
    assert scales[0, 0] == 0x38                   # E4M3(6 / 6) = 1.0
    assert codes[0, 0] == 0xD7                    # ch0 = 6 -> 0x7, ch1 = -3 -> 0xD
    assert codes[0, 1] == 0x02                    # ch2 = 1.25 -> 1.0 (tie to even), ch3 = 0.1 -> 0
    assert codes[0, 2] & 0xF == 0x4               # 2.5 -> 2.0 (tie to even)
    assert scales[0, 1] == 0 and np.all(codes[0, 8:16] == 0)


def test_mxfp4_grid_and_bound():
    g = np.random.default_rng(2)
    x = (g.normal(0, 1, (300, 512)) * g.choice([1e-3, 1, 30], (300, 1))).astype(np.float32)
    codes, scales = F.mxfp4_pack(x)
    assert codes.nbytes // 300 + scales.nbytes // 300 == PAGE["mxfp4_bytes_per_entry_d512"]["value"]
    deq = F.mxfp4_unpack(codes, scales)
    s = np.repeat(F.E4M3_TABLE[scales], 16, axis=1)
    assert np.all(np.abs(deq) <= 6 * s)
    ratio = np.divide(deq, s, out=np.zeros_like(deq), where=s > 0)
    assert np.all(np.isin(np.abs(ratio), np.abs(F.E2M1_TABLE)))
    # the scale is E4M3(amax / 6) of each group
    amax = np.abs(x.reshape(300, 32, 16)).max(axis=2)
    assert np.array_equal(scales, F.e4m3_encode_array((amax / np.float32(6)).astype(np.float32)))
    # error: at most half the widest E2M1 step (1.0 * s) plus what saturation at
    # 6 * s cuts off; a scale that rounds to zero only for amax / 6 <= 2**-10
    err = np.abs(np.abs(x) - np.abs(deq)).reshape(300, 32, 16).max(axis=2)
    sv = F.E4M3_TABLE[scales]
    ok = err <= 1.0 * sv + np.maximum(amax - 6 * sv, 0) + 1e-12
    assert np.all(ok[sv > 0])
    assert np.all(amax[sv == 0] / 6 <= 2.0 ** -10)
    assert (sv == 0).any() and (sv > 0).any()


def test_mxfp4_vectorised_equals_per_row_rule():
    g = np.random.default_rng(4)
    x = (g.normal(0, 2, (40, 64))).astype(np.float32)
    x[3, :16] = 0
    codes, scales = F.mxfp4_pack(x)
    for i in range(40):
        c, s = F.mxfp4_pack_row(x[i])
        assert np.array_equal(c, codes[i]) and np.array_equal(s, scales[i])


def test_mxfp4_every_code_scale_pair_is_exact_in_bf16():
    c4 = np.arange(16, dtype=np.uint8)
    for sc in range(256):
        if np.isnan(F.E4M3_TABLE[sc]):
            continue
        codes = (c4[0::2] | (c4[1::2] << 4)).reshape(1, 8)
        deq = F.mxfp4_unpack(codes, np.array([[sc]], np.uint8))
        assert np.array_equal(deq[0], F.E2M1_TABLE * F.E4M3_TABLE[sc])
        assert np.array_equal(F.bf16_round(deq[0].astype(np.float32)), deq[0])
        assert np.array_equal(deq[0].astype(np.float32).astype(np.float64), deq[0])


def test_fp8_round_trip_all_codes():
    for c in range(256):
        if np.isnan(F.E4M3_TABLE[c]):
            continue
        assert F.e4m3_encode(F.E4M3_TABLE[c]) == c


def test_fp8_window_pack():
    g = np.random.default_rng(5)
    x = g.normal(0, 1, (50, 512)).astype(np.float32)
    x[7] = 0
    codes, s = F.fp8_pack(x)
    amax = np.abs(x).max(axis=1)
    assert np.array_equal(s, (amax / np.float32(448)).astype(np.float32))
    assert np.all(codes[7] == 0) and s[7] == 0
    # the largest element of each row maps to +/-448 (or just below after rounding)
    deq = F.E4M3_TABLE[codes] * s[:, None]
    i = np.argmax(np.abs(x), axis=1)
    top = np.abs(F.E4M3_TABLE[codes[np.arange(50), i]])
    assert np.all(top[np.arange(50) != 7] == 448)
    rel = np.abs(deq - x)[np.arange(50) != 7] / amax[np.arange(50) != 7, None]
    # half the largest E4M3 spacing (32 between 256 and 448) times the scale
    assert rel.max() <= 16.0 / 448.0 * (1 + 1e-6)
    out = F.fp8_unpack_bf16(codes, s)
    assert np.array_equal(F.bf16_round(out.astype(np.float32)), out)
