"""Pins for the oracle's quantizers (CPU only)."""

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import quant as Q
from tests.conftest import read_golden


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def test_constants_match_page():
    g = {k: float(v) for k, v in read_golden("quant_constants.txt")}
    assert Q.FP8_MAX == np.float32(g["fp8_max"])
    assert Q.MIN_SCALE == np.float32(1.0 / g["min_scale_denominator"])


def test_constant_row_maps_to_448():
    x = _bf16(np.array([[1.5] * 64, [-0.3125] * 64]))
    q, s = Q.quant_act(x)
    assert s[0] == np.float32(1.5) / np.float32(448) and s[1] == np.float32(0.3125) / np.float32(448)
    assert np.all(q[0] == 0x7E) and np.all(q[1] == 0xFE)


def test_zero_row_uses_min_scale():
    q, s = Q.quant_act(np.zeros((2, 32), dtype=np.float32))
    assert np.all(s == Q.MIN_SCALE) and np.all(q == 0)


def test_quant_act_matches_torch_fp32_pipeline():
    # Independent implementation: torch's own fp32 ops and its float8 cast.
    rng = np.random.default_rng(2)
    x = rng.standard_normal((64, 512)).astype(np.float32)
    x[:, rng.choice(512, 6, replace=False)] *= 20
    x[5] *= 1e-6
    x = _bf16(x)
    q, s = Q.quant_act(x)
    t = torch.from_numpy(x)
    ts = (t.abs().amax(dim=1, keepdim=True) / 448.0).clamp_min(1.0 / (448.0 * 512.0))
    tq = (t / ts).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(s, ts.reshape(-1).numpy())
    assert np.array_equal(q, tq)


def test_group_quant_is_independent_per_group():
    rng = np.random.default_rng(3)
    x = _bf16(rng.standard_normal((4, 384)))
    x[:, 128:256] *= 50.0
    x = _bf16(x)
    q, s = Q.quant_act(x, group=128)
    assert s.shape == (4, 3)
    for g in range(3):
        qg, sg = Q.quant_act(x[:, g * 128:(g + 1) * 128])
        assert np.array_equal(qg, q[:, g * 128:(g + 1) * 128])
        assert np.array_equal(sg, s[:, g])


def test_quant_act_rejects_nan():
    x = np.ones((1, 32), dtype=np.float32)
    x[0, 3] = np.nan
    with pytest.raises(ValueError):
        Q.quant_act(x)


def test_mxfp4_scale_rule():
    w = np.zeros((1, 128))
    w[0, :32] = np.linspace(-1.0, 1.0, 32)          # amax 1.0 -> X = -2
    w[0, 32:64] = 0.99                             # amax 0.99 -> X = -3, 7.92 saturates to 6
    w[0, 64:96] = 6.0 * 2.0 ** -5                  # exactly representable, X = -5
    packed, sc = Q.quant_mxfp4_ocp(w)              # block 3 all zero
    assert list(sc[0]) == [125, 124, 122, 127]
    codes = F.unpack_e2m1(packed, 128)[0]
    assert codes[31] == 6 and codes[0] == 14       # +1.0 / 0.25 = 4, -1.0 -> -4
    assert np.all(codes[32:64] == 7)               # saturated at 6
    assert np.all(codes[64:96] == 7)               # 6.0 exactly
    assert np.all(codes[96:] == 0)


def test_mxfp4_dequant_quant_idempotent():
    rng = np.random.default_rng(4)
    w = rng.standard_normal((16, 256)) * 0.02
    p1, s1 = Q.quant_mxfp4_ocp(w)
    wd = Q.dequant_mxfp4(p1, s1, 256)
    p2, s2 = Q.quant_mxfp4_ocp(wd)
    assert np.array_equal(p1, p2) and np.array_equal(s1, s2)
    # In units of the block scale 2^X the block's magnitudes lie below 8: the
    # e2m1 grid step is at most 2 (half-step 1), and saturation of (6, 8) to 6
    # costs at most 2.
    err = np.abs(wd - w)
    blk = np.repeat(F.ue8m0_decode(s1), 32, axis=1)
    assert np.all(err <= 2.0 * blk)
    inside = np.abs(w) <= 6.0 * blk
    assert np.all(err[inside] <= blk[inside])


def test_blockfp8_weight_quant():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((256, 256)) * 0.02).astype(np.float32)
    w[128:, 128:] = 0
    codes, s = Q.quant_blockfp8_w(w)
    assert s.shape == (2, 2) and s[1, 1] == 1.0
    amax00 = np.float32(np.max(np.abs(w[:128, :128])))
    assert s[0, 0] == amax00 / np.float32(448)
    i = np.unravel_index(np.argmax(np.abs(w[:128, :128])), (128, 128))
    assert codes[i] & 0x7F == 0x7E
    wd = F.e4m3_decode(codes) * np.repeat(np.repeat(s, 128, 0), 128, 1)
    rel = np.abs(wd - w)[w != 0] / np.abs(w[w != 0])
    big = np.abs(w[w != 0]) > 2.0 ** -6 * np.repeat(np.repeat(s, 128, 0), 128, 1)[w != 0]
    assert np.all(rel[big] <= 2.0 ** -4 + 1e-7)
