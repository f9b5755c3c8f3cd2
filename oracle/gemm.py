"""GEMM definitions (oracle; test infrastructure only).

Every GEMM is written as its plain definition: decode every code by table,
form products and sums in float64, apply the fp32 scales in float64, round once
to bfloat16 (round-to-nearest-even). Work is split over N only (independent
output columns) to bound memory; nothing is reordered within a dot product
beyond what NumPy's float64 matmul does.

Exactness. For the two quantized GEMMs the inner float64 sum is exact:
e4m3 x e2m1 products carry at most 6 significant bits and e4m3 x e4m3 products
at most 8, and for the operand ranges of the workloads the span of product
exponents plus log2(K) stays far below 53 bits. So the summation order cannot
change the result; ``exact_check=True`` asserts that by recomputing with K
reversed and requiring bit-identical float64.
"""

import numpy as np

from .formats import bf16_round, e2m1_decode, e4m3_decode, ue8m0_decode, unpack_e2m1


def _chunks(n, step):
    for a in range(0, n, step):
        yield a, min(n, a + step)


def gemm_w4a8(q, s, w_packed, w_scale, rows=None, chunk=1024, exact_check=False):
    """W4A8 MXFP4 linear: C[m,n] = bf16( s[m] * sum_k e4m3(q[m,k]) * e2m1(w[n,k]) * 2^(e[n,k/32]-127) ).

    radiance_mxfp4.py: module docstring (fp8 activations against e2m1 weights
    with a ue8m0 scale per 32 K) and ``_exact_ref`` (dequantize the weight by
    table, scale the activations by their per-token scale, multiply).

    q: uint8 [M, K] e4m3 codes; s: float32 [M]; w_packed: uint8 [N, K/2]
    (checkpoint order, low nibble = even k); w_scale: uint8 [N, K/32].
    rows: optional index array of output columns n to compute.
    Returns (c64 float64 [M, n], c_bf16 float64 [M, n]) -- the exact value
    before rounding and its bfloat16 rounding.
    """
    q = np.asarray(q, dtype=np.uint8)
    s = np.asarray(s, dtype=np.float32).reshape(-1)
    M, K = q.shape
    A = e4m3_decode(q)
    idx = np.arange(w_packed.shape[0]) if rows is None else np.asarray(rows)
    out = np.empty((M, len(idx)), dtype=np.float64)
    for a, b in _chunks(len(idx), chunk):
        r = idx[a:b]
        W = e2m1_decode(unpack_e2m1(w_packed[r], K)) * np.repeat(ue8m0_decode(w_scale[r]), 32, axis=1)
        acc = A @ W.T
        if exact_check:
            acc_rev = A[:, ::-1] @ W[:, ::-1].T
            if not np.array_equal(acc, acc_rev):
                raise AssertionError("gemm_w4a8: float64 sum is not exact for these inputs")
        out[:, a:b] = s.astype(np.float64)[:, None] * acc
    return out, bf16_round(out)


def gemm_w4a4(x_packed, x_scale, w_packed, w_scale, rows=None, chunk=1024, exact_check=False):
    """W4A4 MXFP4 x MXFP4 (next step; oracle only):
    C[m,n] = bf16( sum_k e2m1(x[m,k]) 2^(a[m,k/32]-127) * e2m1(w[n,k]) 2^(e[n,k/32]-127) ).

    radiance_mxfp4.py: the W4A4 path the page's W4A8 kernel replaces (module
    docstring; ``_debug_compare``). Both operands in checkpoint order (low
    nibble = even k) with one ue8m0 scale per 32 K. e2m1 x e2m1 products carry
    at most 4 significant bits, so the float64 sum is exact for the workloads'
    scale ranges (``exact_check`` re-sums with K reversed).

    Returns (c64 float64 [M, n], c_bf16 float64 [M, n]).
    """
    x_packed = np.asarray(x_packed, dtype=np.uint8)
    M = x_packed.shape[0]
    K = 2 * x_packed.shape[1]
    A = e2m1_decode(unpack_e2m1(x_packed, K)) * np.repeat(ue8m0_decode(x_scale), 32, axis=1)
    idx = np.arange(w_packed.shape[0]) if rows is None else np.asarray(rows)
    out = np.empty((M, len(idx)), dtype=np.float64)
    for a, b in _chunks(len(idx), chunk):
        r = idx[a:b]
        W = e2m1_decode(unpack_e2m1(w_packed[r], K)) * np.repeat(ue8m0_decode(w_scale[r]), 32, axis=1)
        acc = A @ W.T
        if exact_check:
            acc_rev = A[:, ::-1] @ W[:, ::-1].T
            if not np.array_equal(acc, acc_rev):
                raise AssertionError("gemm_w4a4: float64 sum is not exact for these inputs")
        out[:, a:b] = acc
    return out, bf16_round(out)


def gemm_blockfp8(q, As, w, Ws, rows=None, chunk=1024, exact_check=False):
    """Block-FP8 W8A8: C[m,n] = bf16( sum_kb As[m,kb] Ws[n/128,kb] sum_{k in kb} e4m3(q[m,k]) e4m3(w[n,k]) ).

    radiance_kernels.py, ``block_scaled_mm`` (A e4m3 with act scales As, one per
    token per 128 K; B e4m3 with one weight scale per 128x128 block, used as a
    multiplier). The per-block partial sum is exact; the scale products and the
    sum over blocks are float64.

    q: uint8 [M, K]; As: float32 [M, K/128]; w: uint8 [N, K]; Ws: float32
    [N/128, K/128]. Returns (c64, c_bf16) like ``gemm_w4a8``.
    """
    q = np.asarray(q, dtype=np.uint8)
    M, K = q.shape
    KB = K // 128
    A = e4m3_decode(q)
    As = np.asarray(As, dtype=np.float32).astype(np.float64).reshape(M, KB)
    Ws = np.asarray(Ws, dtype=np.float32).astype(np.float64)
    idx = np.arange(w.shape[0]) if rows is None else np.asarray(rows)
    out = np.zeros((M, len(idx)), dtype=np.float64)
    for a, b in _chunks(len(idx), chunk):
        r = idx[a:b]
        W = e4m3_decode(w[r])
        wsr = Ws[r // 128]                                   # [n, KB]
        acc = np.zeros((M, b - a), dtype=np.float64)
        for kb in range(KB):
            sl = slice(kb * 128, (kb + 1) * 128)
            P = A[:, sl] @ W[:, sl].T                        # exact
            if exact_check:
                P2 = A[:, sl][:, ::-1] @ W[:, sl][:, ::-1].T
                if not np.array_equal(P, P2):
                    raise AssertionError("gemm_blockfp8: block sum is not exact")
            acc += (As[:, kb][:, None] * wsr[:, kb][None, :]) * P
        out[:, a:b] = acc
    return out, bf16_round(out)


def gemm_bf16(x, w, rows=None, chunk=4096):
    """Skinny bf16 NT GEMM: C = bf16( x W^T ), products and sum in float64.

    radiance_gemm.py, module docstring: C[M,N] = x[M,K] @ W[N,K]^T with the
    bf16 result of a higher-precision accumulation.

    x: [M, K] and w: [N, K] float arrays holding bfloat16 values.
    Returns (c64, c_bf16).
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    idx = np.arange(w.shape[0]) if rows is None else np.asarray(rows)
    out = np.empty((x.shape[0], len(idx)), dtype=np.float64)
    for a, b in _chunks(len(idx), chunk):
        out[:, a:b] = x @ w[idx[a:b]].T
    return out, bf16_round(out)


def rel_frobenius(out, ref):
    """||out - ref|| / ||ref||: the error measure the radiance_mxfp4.py page
    reports (``_debug_compare``), with 0.02 as its "wrong" threshold."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(out - ref) / max(np.linalg.norm(ref), 1e-30))


def gemm_tolerance_ok(out, ref):
    """Elementwise acceptance: |out - ref| <= 4e-3 |ref| + 1e-3 rms(ref row).

    Returns (ok: bool, worst ratio of error to bound).
    """
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    bound = 4e-3 * np.abs(ref) + 1e-3 * rms
    err = np.abs(out - ref)
    ratio = np.max(err / np.maximum(bound, 1e-300)) if err.size else 0.0
    return bool(np.all(err <= bound)), float(ratio)
