"""Pins for the oracle's GEMM definitions: one-hot weights, exact brute force
with rational arithmetic, invariants (CPU only)."""

from fractions import Fraction

import numpy as np

from oracle import formats as F
from oracle import gemm as G
from oracle import quant as Q


def _frac_e4m3(c):
    return Fraction(F.E4M3_VALUES[int(c)])


def test_w4a8_one_hot_weights():
    rng = np.random.default_rng(10)
    M, N, K = 3, 5, 128
    q = rng.integers(0, 0x7E, (M, K)).astype(np.uint8)
    s = rng.uniform(0.001, 0.01, M).astype(np.float32)
    codes = np.zeros((N, K), dtype=np.uint8)
    scale = np.full((N, K // 32), 127, dtype=np.uint8)
    # (n, k, e2m1 code, scale code) -- odd and even k, several 32-blocks, negative code
    spots = [(0, 0, 3, 127), (1, 33, 7, 120), (2, 64, 13, 130), (3, 127, 1, 100), (4, 94, 10, 127)]
    for n, k, c, e in spots:
        codes[n, k] = c
        scale[n, k // 32] = e
    packed = F.pack_e2m1(codes)
    c64, cb = G.gemm_w4a8(q, s, packed, scale)
    for n, k, c, e in spots:
        want = s.astype(np.float64) * F.e4m3_decode(q[:, k]) * F.E2M1_VALUES[c] * 2.0 ** (e - 127)
        assert np.array_equal(c64[:, n], want)
        assert np.array_equal(cb[:, n], F.bf16_round(want))


def test_w4a8_brute_force_rational():
    rng = np.random.default_rng(11)
    M, N, K = 3, 4, 64
    q = rng.integers(0, 0xFE, (M, K)).astype(np.uint8)
    q[q == 0x7F] = 0x10
    s = rng.uniform(1e-3, 1e-2, M).astype(np.float32)
    codes = rng.integers(0, 16, (N, K)).astype(np.uint8)
    scale = rng.integers(115, 135, (N, K // 32)).astype(np.uint8)
    c64, cb = G.gemm_w4a8(q, s, F.pack_e2m1(codes), scale)
    for m in range(M):
        for n in range(N):
            acc = sum(_frac_e4m3(q[m, k]) * Fraction(F.E2M1_VALUES[codes[n, k]])
                      * Fraction(2) ** (int(scale[n, k // 32]) - 127) for k in range(K))
            exact = Fraction(float(s[m])) * acc
            assert c64[m, n] == float(exact)          # one rounding (fp64) of the exact value
            assert cb[m, n] == F.bf16_round(np.array([float(exact)]))[0]


def test_w4a8_sum_is_exact_on_workload_like_data():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((8, 2048)) * 1.0).astype(np.float32)
    q, s = Q.quant_act(x)
    w = rng.standard_normal((64, 2048)) * 0.02
    p, sc = Q.quant_mxfp4_ocp(w)
    G.gemm_w4a8(q, s, p, sc, exact_check=True)


def test_w4a8_scale_code_linearity():
    rng = np.random.default_rng(13)
    q = rng.integers(0, 0x7E, (2, 64)).astype(np.uint8)
    s = np.array([0.01, 0.02], dtype=np.float32)
    p = rng.integers(0, 256, (3, 32)).astype(np.uint8)
    sc = rng.integers(110, 130, (3, 2)).astype(np.uint8)
    a, _ = G.gemm_w4a8(q, s, p, sc)
    b, _ = G.gemm_w4a8(q, s, p, sc + 1)
    assert np.array_equal(b, 2 * a)


def test_w4a8_rows_subset_matches_full():
    rng = np.random.default_rng(14)
    q = rng.integers(0, 0x7E, (4, 64)).astype(np.uint8)
    s = np.ones(4, dtype=np.float32)
    p = rng.integers(0, 256, (9, 32)).astype(np.uint8)
    sc = rng.integers(120, 130, (9, 2)).astype(np.uint8)
    full, _ = G.gemm_w4a8(q, s, p, sc, chunk=4)
    sub, _ = G.gemm_w4a8(q, s, p, sc, rows=np.array([1, 5, 8]))
    assert np.array_equal(full[:, [1, 5, 8]], sub)


def test_blockfp8_unit_scales_is_plain_e4m3_dot():
    rng = np.random.default_rng(15)
    M, N, K = 2, 3, 256
    q = rng.integers(0, 0x7E, (M, K)).astype(np.uint8)
    w = rng.integers(0x80, 0xFE, (N, K)).astype(np.uint8)
    c64, _ = G.gemm_blockfp8(q, np.ones((M, 2), np.float32), w, np.ones((1, 2), np.float32))
    for m in range(M):
        for n in range(N):
            exact = sum(_frac_e4m3(q[m, k]) * _frac_e4m3(w[n, k]) for k in range(K))
            assert c64[m, n] == float(exact)


def test_blockfp8_scale_placement_one_hot():
    M, N, K = 2, 256, 384
    q = np.zeros((M, K), np.uint8)
    w = np.zeros((N, K), np.uint8)
    q[:, 130] = 0x38          # 1.0 in k-block 1
    q[:, 300] = 0x40          # 2.0 in k-block 2
    w[200, 130] = 0x38        # n-block 1
    w[7, 300] = 0x30          # 0.5, n-block 0
    As = np.array([[1, 3, 5], [2, 7, 11]], np.float32)
    Ws = np.array([[13, 17, 19], [23, 29, 31]], np.float32)
    c64, _ = G.gemm_blockfp8(q, As, w, Ws)
    assert c64[0, 200] == 1 * 1 * 3 * 29 and c64[1, 200] == 7 * 29
    assert c64[0, 7] == 2 * 0.5 * 5 * 19 and c64[1, 7] == 11 * 19
    assert np.count_nonzero(c64) == 4


def test_blockfp8_rational_with_scales():
    rng = np.random.default_rng(16)
    M, N, K = 2, 128, 256
    q = rng.integers(0, 0x7E, (M, K)).astype(np.uint8)
    w = rng.integers(0, 0xFE, (N, K)).astype(np.uint8)
    w[w == 0x7F] = 0
    As = rng.uniform(0.01, 0.1, (M, 2)).astype(np.float32)
    Ws = rng.uniform(1e-4, 1e-3, (1, 2)).astype(np.float32)
    c64, _ = G.gemm_blockfp8(q, As, w, Ws, exact_check=True)
    for m in range(M):
        for n in (0, 77, 127):
            exact = Fraction(0)
            for kb in range(2):
                part = sum(_frac_e4m3(q[m, k]) * _frac_e4m3(w[n, k]) for k in range(kb * 128, kb * 128 + 128))
                exact += Fraction(float(As[m, kb])) * Fraction(float(Ws[0, kb])) * part
            assert abs(c64[m, n] - float(exact)) <= 1e-15 * abs(float(exact)) + 1e-300


def test_bf16_gemm_rational():
    rng = np.random.default_rng(17)
    x = torch_bf16(rng.standard_normal((3, 96)))
    w = torch_bf16(rng.standard_normal((5, 96)) * 0.02)
    c64, cb = G.gemm_bf16(x, w)
    for m in range(3):
        for n in range(5):
            exact = sum(Fraction(float(x[m, k])) * Fraction(float(w[n, k])) for k in range(96))
            assert abs(c64[m, n] - float(exact)) <= 2.0 ** -45 * max(abs(float(exact)), 1e-30)
            assert cb[m, n] == F.bf16_round(np.array([float(exact)]))[0]


def torch_bf16(a):
    import torch
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


def test_tolerance_rule():
    rng = np.random.default_rng(18)
    ref = rng.standard_normal((4, 100))
    ok, _ = G.gemm_tolerance_ok(F.bf16_round(ref), ref)
    assert ok
    ok, ratio = G.gemm_tolerance_ok(ref * 1.01, ref)
    assert not ok and ratio > 1
    assert G.rel_frobenius(F.bf16_round(ref), ref) < 0.003


def test_planted_nibble_swap_is_caught():
    """A plausible oracle mistake (reading the high nibble as the even element)
    must break the one-hot pin: planted here on the CPU, in a copy."""
    codes = np.zeros((1, 64), np.uint8)
    codes[0, 1] = 7                                   # odd k
    packed = F.pack_e2m1(codes)
    bad = ((packed & 0x0F) << 4) | (packed >> 4)      # swapped nibbles
    q = np.zeros((1, 64), np.uint8)
    q[0, 1] = 0x38
    good, _ = G.gemm_w4a8(q, np.ones(1, np.float32), packed, np.full((1, 2), 127, np.uint8))
    wrong, _ = G.gemm_w4a8(q, np.ones(1, np.float32), bad, np.full((1, 2), 127, np.uint8))
    assert good[0, 0] == 6.0 and wrong[0, 0] != 6.0
