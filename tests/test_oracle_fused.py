"""Pins for the fused quantization producers of the oracle (CPU only).

Each pin reaches the oracle's result by a route other than its own formula:
closed forms, invariants of RMS normalization and of SiLU, and library
routines (torch CPU bfloat16 addition, torch's SiLU in float64)."""

import numpy as np
import torch

from oracle import formats as F
from oracle import fused as U
from oracle import quant as Q


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return _bf16((torch.randn(*shape, generator=g) * scale).numpy())


def test_residual_add_matches_torch_bf16_add():
    y = _rand((16, 256), 1)
    r = _rand((16, 256), 2, scale=37.0)
    # wide exponent gaps as well: the float32 sum rounds before the bf16 rounding
    r[0] = _bf16(np.ldexp(1.0, np.arange(256) % 40 - 20) * (1 + (np.arange(256) % 7) / 8))
    got, _ = U.add_rmsnorm(y, r, np.zeros(256), 1e-6)
    ref = (torch.from_numpy(y).to(torch.bfloat16) + torch.from_numpy(r).to(torch.bfloat16)).double().numpy()
    assert np.array_equal(got, ref)


def test_constant_row_closed_form():
    """A constant row c with residual 0, weight w: h = sign(c) (1 + w) / sqrt(1 + eps/c^2)."""
    K, c, eps = 128, _bf16(0.75)[()], 1e-6
    y = np.full((1, K), c)
    w = _rand((K,), 3, scale=0.1)
    _, h64 = U.add_rmsnorm(y, np.zeros((1, K)), w, eps)
    exp = (1.0 + w) / np.sqrt(1.0 + np.float64(np.float32(eps)) / (c * c))
    assert np.allclose(h64[0], exp, rtol=1e-15, atol=0)


def test_rms_normalization_invariants():
    """(a) The normalized row has mean square var / (var + eps); (b) scaling the
    input by a power of two leaves h unchanged when eps = 0."""
    K = 512
    y = _rand((4, K), 5)
    w = np.zeros(K)
    r, h64 = U.add_rmsnorm(y, np.zeros_like(y), w, 1e-5)
    var = np.mean(r * r, axis=1)
    ms = np.mean(h64 * h64, axis=1)
    assert np.allclose(ms, var / (var + np.float64(np.float32(1e-5))), rtol=1e-12)
    _, h0 = U.add_rmsnorm(y, np.zeros_like(y), w, 0.0)
    _, h1 = U.add_rmsnorm(np.ldexp(y, 7), np.zeros_like(y), w, 0.0)
    assert np.array_equal(h0, h1)


def test_add_rmsnorm_quant_constant_row_codes():
    """w = 0, a constant row: every h is the same value v, so amax = |v| and
    every code is +-448 (0x7E / 0xFE), s = bf16(v) / 448."""
    K = 64
    y = np.concatenate([np.full((1, K), 3.0), np.full((1, K), -0.125)])
    q, s, r, h64 = U.add_rmsnorm_quant(y, np.zeros_like(y), np.zeros(K), 1e-6)
    assert np.all(q[0] == 0x7E) and np.all(q[1] == 0xFE)
    v = F.bf16_round(h64[:, 0])
    assert np.array_equal(s, (np.abs(v).astype(np.float32) / np.float32(448)).astype(np.float32))


def test_silu_identities_and_library():
    g = _rand((8, 64), 7, scale=3.0)
    gu = np.concatenate([g, np.ones_like(g)], axis=1)
    a, h64 = U.silu_mul(gu)
    ref = torch.nn.functional.silu(torch.from_numpy(g)).numpy()     # float64 library routine
    assert np.array_equal(a, F.bf16_round(ref))
    assert np.array_equal(h64, a)                                     # u = 1
    # silu(x) - silu(-x) = x, in float64 before rounding
    s_pos = g / (1.0 + np.exp(-g))
    s_neg = -g / (1.0 + np.exp(g))
    assert np.allclose(s_pos - s_neg, g, rtol=1e-14, atol=1e-300)
    a0, _ = U.silu_mul(np.zeros((1, 4)))
    assert np.all(a0 == 0)


def test_silu_mul_product_is_exact_before_rounding():
    """bf16 x bf16 products carry <= 16 significant bits, so h64 is the exact
    product and h = bf16(h64) is the single rounding of torch's bf16 multiply."""
    gu = np.concatenate([_rand((4, 32), 11, 2.0), _rand((4, 32), 12, 5.0)], axis=1)
    a, h64 = U.silu_mul(gu)
    u = gu[:, 32:]
    ref = (torch.from_numpy(a).to(torch.bfloat16) * torch.from_numpy(u).to(torch.bfloat16)).double().numpy()
    assert np.array_equal(F.bf16_round(h64), ref)


def test_silu_mul_quant_uses_the_token_rule():
    gu = np.concatenate([_rand((3, 48), 13, 2.0), _rand((3, 48), 14)], axis=1)
    q, s, a, h64 = U.silu_mul_quant(gu)
    q2, s2 = Q.quant_act(F.bf16_round(h64))
    assert np.array_equal(q, q2) and np.array_equal(s, s2)
