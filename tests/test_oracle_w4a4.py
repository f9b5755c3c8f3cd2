"""Pins for the W4A4 oracle (MXFP4 activations x MXFP4 weights), the next
step after the W4A8 path: checked against rational arithmetic, against the
W4A8 definition on operands both formats represent exactly, on one-hot
activations, and for the activation quantizer's round trip."""

from fractions import Fraction

import numpy as np

from oracle import formats as F
from oracle import gemm as G
from oracle import quant as Q


def _rand_mx(rows, K, rng, lo=118, hi=130):
    codes = rng.integers(0, 16, size=(rows, K)).astype(np.uint8)
    return F.pack_e2m1(codes), rng.integers(lo, hi, size=(rows, K // 32)).astype(np.uint8), codes


def test_w4a4_brute_force_rational():
    rng = np.random.default_rng(41)
    M, N, K = 3, 4, 64
    xp, xs, xc = _rand_mx(M, K, rng)
    wp, ws, wc = _rand_mx(N, K, rng)
    c64, cbf = G.gemm_w4a4(xp, xs, wp, ws, exact_check=True)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(F.E2M1_VALUES[xc[m, k]]) * Fraction(2) ** (int(xs[m, k // 32]) - 127)
                        * Fraction(F.E2M1_VALUES[wc[n, k]]) * Fraction(2) ** (int(ws[n, k // 32]) - 127)
                        for k in range(K))
            assert c64[m, n] == float(exact)
            assert cbf[m, n] == F.bf16_round(np.array([float(exact)]))[0]


def test_w4a4_equals_w4a8_on_common_operands():
    """Activations whose blocks of a row share one power-of-two scale are
    exactly an e4m3 tensor with that per-token scale (every e2m1 value is an
    e4m3 value): both definitions must give the identical result."""
    rng = np.random.default_rng(42)
    M, N, K = 5, 7, 256
    xc = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    row_code = rng.integers(118, 132, size=M).astype(np.uint8)
    xs = np.repeat(row_code[:, None], K // 32, axis=1)
    wp, ws, _ = _rand_mx(N, K, rng)
    q = F.e4m3_encode_rne_sat(F.e2m1_decode(xc).astype(np.float32))
    assert np.array_equal(F.e4m3_decode(q), F.e2m1_decode(xc)), "e2m1 values must be exact in e4m3"
    s = np.ldexp(np.float32(1.0), row_code.astype(np.int64) - 127).astype(np.float32)
    a64, _ = G.gemm_w4a4(F.pack_e2m1(xc), xs, wp, ws, exact_check=True)
    b64, _ = G.gemm_w4a8(q, s, wp, ws, exact_check=True)
    assert np.array_equal(a64, b64)


def test_w4a4_one_hot_activation():
    """One nonzero activation code per token, at a token-dependent k (odd and
    even, different 32-blocks), with its own block scale: C[m, n] is that
    element times column k of the dequantized weight."""
    rng = np.random.default_rng(43)
    M, N, K = 6, 9, 128
    xc = np.zeros((M, K), dtype=np.uint8)
    xs = np.full((M, K // 32), 127, dtype=np.uint8)
    ks = [0, 1, 33, 66, 127, 95]
    vals = [1, 9, 7, 15, 4, 3]                 # e2m1 codes, negatives included
    for m, (k, v) in enumerate(zip(ks, vals)):
        xc[m, k] = v
        xs[m, k // 32] = 125 + m
    wp, ws, _ = _rand_mx(N, K, rng)
    W = Q.dequant_mxfp4(wp, ws, K)
    c64, _ = G.gemm_w4a4(F.pack_e2m1(xc), xs, wp, ws)
    for m, (k, v) in enumerate(zip(ks, vals)):
        want = F.E2M1_VALUES[v] * 2.0 ** (125 + m - 127) * W[:, k]
        assert np.array_equal(c64[m], want)


def test_activation_mx_quant_round_trip():
    """Values already on the MX grid (e2m1 value x a power of two, each
    32-block's maximum setting its scale) quantize back to themselves."""
    rng = np.random.default_rng(44)
    M, K = 4, 128
    xc = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    xc[:, ::32] = 7                            # each block's maximum is 6.0
    X = rng.integers(-6, 4, size=(M, K // 32))
    x = F.e2m1_decode(xc) * np.repeat(np.ldexp(1.0, X), 32, axis=1)
    packed, scale = Q.quant_act_mxfp4(x)
    assert np.array_equal(scale, (X + 127).astype(np.uint8))
    assert np.array_equal(Q.dequant_mxfp4(packed, scale, K), x)
