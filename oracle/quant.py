"""Quantizers (oracle; test infrastructure only).

quant_act          -- the method's activation quantization (per token, or per
                      token per 128-K group). The GPU must match it bit for bit.
quant_mxfp4_ocp    -- OCP MX FP4 weight quantization. The pages only ever load
                      pre-quantized checkpoints, so this exists to manufacture
                      test weights.
quant_blockfp8_w   -- 128x128 block e4m3 weight quantization; test inputs only.
"""

import numpy as np

from .formats import (E2M1_MAX, E4M3_MAX, e2m1_encode_rne_sat,
                      e4m3_encode_rne_sat, pack_e2m1)

# radiance_mxfp4.py, comment above ``_traced_quant``: the scale is
# max(rowamax/448, 1/(448*512)), computed in fp32.
FP8_MAX = np.float32(448.0)
MIN_SCALE = np.float32(1.0 / (448.0 * 512.0))


def quant_act(x, group=None):
    """Dynamic e4m3 quantization of activations.

    radiance_mxfp4.py, ``_traced_quant`` and the comment above it: per row
    s = max(amax(|x|) / 448, 1/(448*512)) in fp32, then q = e4m3(clamp(x / s,
    -448, 448)) with round-to-nearest. The plainest reading of "fp32 math" is
    taken: s is the correctly rounded fp32 quotient amax/448 (the form the
    PURE_QUANT branch of ``mxfp4_linear`` writes), and each x/s is a correctly
    rounded fp32 division; the clamp is saturation of finite values.

    With ``group`` = g (block-FP8 activations, radiance_kernels.py
    ``block_scaled_mm``), the same rule runs independently on every g-wide
    slice of each row, giving one scale per token per g of K.

    x: [M, K] float array whose values are bfloat16 numbers.
    Returns (q uint8 [M, K], s float32 [M] or [M, K/g]).
    """
    x = np.asarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("quant_act: non-finite activation (behaviour unspecified)")
    M, K = x.shape
    g = K if group is None else int(group)
    if K % g:
        raise ValueError("quant_act: K must be a multiple of the group")
    xg = x.reshape(M, K // g, g)
    amax = np.max(np.abs(xg), axis=2)                       # exact in fp32
    s = (amax / FP8_MAX).astype(np.float32)                 # fp32 RNE division
    s = np.maximum(s, MIN_SCALE).astype(np.float32)
    y = (xg / s[:, :, None]).astype(np.float32)             # fp32 RNE division
    q = e4m3_encode_rne_sat(y).reshape(M, K)
    if group is None:
        return q, s.reshape(M)
    return q, s


def quant_mxfp4_ocp(w):
    """OCP MX v1.0 FP4 quantization of a weight matrix (test inputs only).

    Per 32-element block of each row: X = floor(log2(amax)) - 2 (2 is the
    largest e2m1 exponent), scale code X + 127 clamped to [0, 254]; elements
    e2m1_rne_sat(w / 2^X). An all-zero block gets code 127. Packed two codes per
    byte, low nibble = even k, as the radiance_mxfp4.py page reads them.

    w: [N, K] float. Returns (packed uint8 [N, K/2], scale uint8 [N, K/32]).
    """
    w = np.asarray(w, dtype=np.float64)
    N, K = w.shape
    if K % 32:
        raise ValueError("quant_mxfp4_ocp: K must be a multiple of 32")
    wb = w.reshape(N, K // 32, 32)
    amax = np.max(np.abs(wb), axis=2)
    _, e = np.frexp(amax)                   # amax = m 2^e, 0.5 <= m < 1
    X = np.where(amax > 0, (e - 1) - 2, 0)  # floor(log2(amax)) - emax(e2m1)
    code = np.clip(X + 127, 0, 254)
    X = code - 127
    y = np.ldexp(wb, -X[:, :, None])        # exact power-of-two scaling
    codes = e2m1_encode_rne_sat(y).reshape(N, K)
    return pack_e2m1(codes), code.astype(np.uint8)


def quant_act_mxfp4(x):
    """MXFP4 activations for the W4A4 variant (next step; oracle only).

    radiance_mxfp4.py names the W4A4 path only as the library fallback that
    quantizes activations to MXFP4 (module docstring; ``_debug_compare``,
    "aiter quantizes x to mxfp4") and prints neither its rule nor its kernel.
    Reading taken: the OCP MX v1.0 rule the weights follow, per 32-element
    block along K of each token -- X = floor(log2 amax) - 2, scale code X + 127
    clamped to [0, 254], elements e2m1_rne_sat(x / 2^X), an all-zero block
    code 127 (``quant_mxfp4_ocp``).

    x: [M, K] float (bf16 values). Returns (packed uint8 [M, K/2], scale uint8 [M, K/32]).
    """
    return quant_mxfp4_ocp(x)


def quant_blockfp8_w(w, block=128):
    """Block e4m3 weight quantization (test inputs only).

    Per 128x128 block: s = amax/448 in fp32 (s = 1 for an all-zero block),
    q = e4m3_rne_sat(w / s) with fp32 division. The scale is a multiplier,
    w ~ q * s (radiance_kernels.py names it ``weight_scale_inv`` but passes it
    to the GEMM as the dequantization multiplier).

    w: [N, K] float with N, K multiples of 128.
    Returns (codes uint8 [N, K], scales float32 [N/128, K/128]).
    """
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    if N % block or K % block:
        raise ValueError("quant_blockfp8_w: N and K must be multiples of 128")
    wb = w.reshape(N // block, block, K // block, block)
    amax = np.max(np.abs(wb), axis=(1, 3))
    s = (amax / FP8_MAX).astype(np.float32)
    s = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    y = (wb / s[:, None, :, None]).astype(np.float32)
    codes = e4m3_encode_rne_sat(y).reshape(N, K)
    return codes, s


def dequant_mxfp4(packed, scale, K):
    """Checkpoint-order MXFP4 -> float64 [N, K] (used by the GEMM definition)."""
    from .formats import e2m1_decode, ue8m0_decode, unpack_e2m1
    codes = unpack_e2m1(packed, K)
    sc = ue8m0_decode(scale)                       # [N, K/32]
    return e2m1_decode(codes) * np.repeat(sc, 32, axis=1)


__all__ = ["quant_act", "quant_mxfp4_ocp", "quant_act_mxfp4", "quant_blockfp8_w", "dequant_mxfp4",
           "FP8_MAX", "MIN_SCALE", "E2M1_MAX", "E4M3_MAX"]
