"""Pins for the oracle's number formats against the pages, library routines
and closed forms (CPU only)."""

import math

import numpy as np
import pytest
import torch

from oracle import formats as F
from tests.conftest import read_golden


def test_e2m1_table_matches_page():
    rows = read_golden("e2m1_table.txt")
    assert len(rows) == 16
    for code, val in rows:
        v = float(val)
        got = F.E2M1_VALUES[int(code)]
        assert got == v and math.copysign(1, got) == math.copysign(1, v)


def test_e2m1_table_matches_ocp_closed_form():
    # OCP MX FP4 E2M1: bias 1, subnormal when the exponent field is 0.
    for c in range(16):
        s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
        mag = (m * 0.5) if e == 0 else (1 + m * 0.5) * 2.0 ** (e - 1)
        assert F.E2M1_VALUES[c] == (-mag if s else mag)


def test_e4m3_table_matches_torch():
    codes = torch.arange(256, dtype=torch.int64).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.E4M3_VALUES
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ref[~nan], ours[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x38] == 1.0


def _torch_e4m3(v32):
    t = torch.from_numpy(np.asarray(v32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encoder_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = F.e4m3_encode_rne_sat(F.e4m3_decode(codes))
    assert np.array_equal(back, codes)


def test_e4m3_encoder_matches_torch_on_random_and_midpoints():
    rng = np.random.default_rng(0)
    v = rng.standard_normal(200000).astype(np.float32) * np.float32(64.0)
    v = np.clip(v, -448, 448).astype(np.float32)
    tiny = (rng.standard_normal(20000) * 2.0 ** -8).astype(np.float32)
    pos = np.sort(F.E4M3_VALUES[:0x7F])
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)     # exact in fp32
    allv = np.concatenate([v, tiny, mids, -mids])
    assert np.array_equal(F.e4m3_encode_rne_sat(allv), _torch_e4m3(allv))


def test_e4m3_encoder_saturates_and_signs():
    got = F.e4m3_encode_rne_sat(np.array([448.0, 460.0, 1e6, -1e6, -0.0, -1e-9, 0.0]))
    assert list(got) == [0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x80, 0x00]
    with pytest.raises(ValueError):
        F.e4m3_encode_rne_sat(np.array([np.nan]))


def test_e2m1_encoder_roundtrip_ties_saturation():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(F.e2m1_encode_rne_sat(F.e2m1_decode(codes)), codes)
    # Round-half-to-even on the e2m1 grid 0, .5, 1, 1.5, 2, 3, 4, 6: each
    # midpoint goes to the neighbour whose mantissa bit is 0 (even code).
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6,
             0.26: 1, 0.74: 1, 2.51: 5, 4.99: 6, 5.01: 7,
             7.0: 7, 100.0: 7, -0.25: 8, -5.0: 14, -100.0: 15}
    for v, c in cases.items():
        assert F.e2m1_encode_rne_sat(np.array([v]))[0] == c, v


def test_ue8m0_decode():
    got = F.ue8m0_decode(np.array([127, 128, 126, 0, 254, 255]))
    assert got[0] == 1.0 and got[1] == 2.0 and got[2] == 0.5
    assert got[3] == 2.0 ** -127 and got[4] == 2.0 ** 127 and np.isnan(got[5])


def test_nibble_order_matches_page():
    for bhex, even, odd in read_golden("nibble_order.txt"):
        b = np.array([[int(bhex, 16)]], dtype=np.uint8)
        assert list(F.unpack_e2m1(b, 2)[0]) == [int(even), int(odd)]
        assert F.pack_e2m1(np.array([[int(even), int(odd)]]))[0, 0] == int(bhex, 16)


def test_bf16_round_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(100000) * 10.0,
        rng.standard_normal(1000) * 1e-38,       # bf16 subnormal range
        np.clip(rng.standard_normal(1000), -3, 3) * 1e38,  # near overflow
    ]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    ours = F.bf16_round(v.astype(np.float64))
    assert np.array_equal(ref, ours)


def test_bf16_round_is_a_single_rounding():
    # 1 + 2^-8 + 2^-30 lies just above the midpoint between 1 and 1 + 2^-7.
    # Direct rounding goes up; rounding through float32 first would lose the
    # 2^-30 and tie back down to 1.0.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert F.bf16_round(np.array([v]))[0] == 1.0 + 2.0 ** -7
    assert F.bf16_round(np.array([1.0 + 2.0 ** -8]))[0] == 1.0          # tie -> even
    assert F.bf16_round(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6
    assert F.bf16_round(np.array([2.0 ** 128]))[0] == np.inf
    assert F.bf16_round(np.array([F.BF16_MAX]))[0] == F.BF16_MAX


def test_bf16_bits_roundtrip():
    vals = F.bf16_round(np.array([1.0, -2.5, 3.14159, 1e-30, 6e37]))
    assert np.array_equal(F.bf16_from_bits(F.bf16_bits(vals)), vals)
