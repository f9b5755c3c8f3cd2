"""Fused quantization producers (oracle; test infrastructure only).

radiance_arnq.py replaces two standalone epilogues that feed a W4A8 linear
with one kernel each, keeping the (q e4m3, per-token fp32 scale) contract of
the per-token quantization:

  * ``ar_add_rms_quant`` (module docstring, "residual add + Gemma rms_norm ->
    per-token fp8 quant"): returns the codes, the scales and the new residual;
  * ``silu_mul_quant`` (the ``_SiluMulQuant`` docstring: a drop-in for the
    MLP's SiluAndMul that returns (q_fp8, scale)).

The pages name these chains but print neither the norm nor the activation, so
the plainest readings of the named operations are taken (each listed in the
design notes):

  * residual add: the two bfloat16 tensors are added in float32 and the sum is
    rounded once to bfloat16; that sum is both the new residual and the norm's
    input;
  * Gemma RMS norm: h = r / sqrt(mean_k(r^2) + eps) * (1 + w), the weight
    offset by one, formed from the bfloat16 r and w and rounded once to
    bfloat16 (here: every product and sum in float64, eps the float32 value);
  * SiluAndMul on [g | u] (each half N wide): a = bfloat16(g * sigmoid(g)),
    h = bfloat16(a * u);
  * then the per-token quantization of h (``quant.quant_act``).

Each function also returns the float64 value of h before its bfloat16
rounding, so a test can tell a rounding-boundary case from an error.
"""

import numpy as np

from .formats import bf16_round
from .quant import quant_act


def add_rmsnorm(y, residual, w, eps):
    """r = bf16(f32(y) + f32(residual)); h64 = r / sqrt(mean(r^2) + eps) * (1 + w).

    y, residual: [M, K] bfloat16 values; w: [K] bfloat16 values; eps: float.
    Returns (r float64 [M, K] (bfloat16 values), h64 float64 [M, K]).
    """
    y32 = np.asarray(y, dtype=np.float32)
    r32 = np.asarray(residual, dtype=np.float32)
    r = bf16_round((y32 + r32).astype(np.float64))        # one float32 add, one bf16 rounding
    var = np.mean(r * r, axis=1, keepdims=True)            # r^2 exact in float64
    inv = 1.0 / np.sqrt(var + np.float64(np.float32(eps)))
    wd = np.asarray(w, dtype=np.float64)
    h64 = r * inv * (1.0 + wd)[None, :]
    return r, h64


def add_rmsnorm_quant(y, residual, w, eps):
    """radiance_arnq.py, ``ar_add_rms_quant`` (single-rank epilogue):
    (q, s, r) = quant(bf16(RMSNorm_gemma(bf16(y + residual)))), r.

    Returns (q uint8 [M, K], s float32 [M], r float64 [M, K], h64 float64 [M, K]).
    """
    r, h64 = add_rmsnorm(y, residual, w, eps)
    h = bf16_round(h64)
    if not np.all(np.isfinite(h)):
        raise ValueError("add_rmsnorm_quant: non-finite normalized value")
    q, s = quant_act(h)
    return q, s, r, h64


def silu_mul(gu):
    """SiluAndMul on [g | u]: h64 = bf16(g * sigmoid(g)) * u (exact product).

    gu: [M, 2N] bfloat16 values. Returns (a float64 [M, N] (bfloat16 values),
    h64 float64 [M, N] before the final bfloat16 rounding).
    """
    gu = np.asarray(gu, dtype=np.float64)
    N = gu.shape[1] // 2
    g, u = gu[:, :N], gu[:, N:]
    with np.errstate(over="ignore"):
        a64 = g / (1.0 + np.exp(-g))
    a = bf16_round(a64)
    return a, a * u


def silu_mul_quant(gu):
    """radiance_arnq.py, ``silu_mul_quant``: (q, s) = quant(bf16(bf16(silu(g)) * u)).

    Returns (q uint8 [M, N], s float32 [M], a float64 [M, N], h64 float64 [M, N]).
    """
    a, h64 = silu_mul(gu)
    h = bf16_round(h64)
    if not np.all(np.isfinite(h)):
        raise ValueError("silu_mul_quant: non-finite activation")
    q, s = quant_act(h)
    return q, s, a, h64
