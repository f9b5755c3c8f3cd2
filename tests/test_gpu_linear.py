"""GPU parity: r4_linear_w4a8_mxfp4, per-token quantization + W4A8 GEMM from
bf16 activations in one call (the quantization kernel into the workspace,
then the GEMM). Its result must equal r4_quant_fp8_per_token followed by
r4_gemm_w4a8_mxfp4 bit for bit, and the oracle's quantize-then-GEMM within
the GEMM tolerance."""

import numpy as np
import pytest
import torch

from block_scaled_precision_token_gb300 import synth
from oracle import gemm as G
from oracle import quant as Q
from tests.gpu_util import assert_gemm_matches, check_device_error, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def r4q():
    m = require_gpu()
    yield m


def _weights(r4q, N, K, seed=0):
    w = synth.weights_fp32(N, K, synth.CFG_DECODE)
    if seed:
        w = w * (1.0 + 0.25 * torch.from_numpy(np.random.default_rng(seed).standard_normal(w.shape)).float())
    p, sc = Q.quant_mxfp4_ocp(w.numpy())
    pk = r4q.prepack_mxfp4(torch.from_numpy(p).cuda(), torch.from_numpy(sc).cuda(), N, K)
    return pk, p, sc


def _linear(r4q, x, pk, N, K, ldc=None):
    """x: bf16 [M, >= K] on the GPU (row stride x.stride(0))."""
    M = x.shape[0]
    full = None
    out = None
    if ldc is not None:
        full = torch.full((M + 2, ldc), 7.0, dtype=torch.bfloat16, device="cuda")
        out = full[:M, :N]
    ws = r4q.workspace(r4q.R4_OP_LINEAR_W4A8_MXFP4, M, N, K)
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda") if out is None else out
    r4q.r4_linear_w4a8_mxfp4(x, x.stride(0), pk, M, N, K, c, c.stride(0), ws)
    check_device_error(r4q)
    return c, full


@pytest.mark.parametrize("N,K", [(384, 1024), (300, 416), (2048, 5120), (5120, 17408), (34816, 5120)])
@pytest.mark.parametrize("M", [1, 6, 16, 33, 64])
def test_equals_quant_then_gemm(r4q, M, N, K):
    """Every token-tile size (16/32/64), a partial last K block (K = 416),
    split-K schedules (5120 x 17408): exactly the bits of quantizing first."""
    pk, _, _ = _weights(r4q, N, K)
    x = synth.activations(M, K, synth.CFG_DECODE, outliers=True).cuda()
    c, _ = _linear(r4q, x, pk, N, K)
    q, s = r4q.quant_fp8(x)
    ref = r4q.gemm_w4a8(q, s, pk, N, K)
    check_device_error(r4q)
    assert torch.equal(c, ref)


@pytest.mark.parametrize("M,N,K", [(6, 640, 1792), (16, 2048, 5120), (11, 5120, 17408)])
def test_against_oracle(r4q, M, N, K):
    pk, p, sc = _weights(r4q, N, K, seed=M)
    x = synth.activations(M, K, synth.CFG_DECODE, outliers=True)
    c, _ = _linear(r4q, x.cuda(), pk, N, K)
    q, s = Q.quant_act(x.float().numpy())
    rows = None if N <= 2048 else synth.sample_indices(N, 384, M).numpy()
    c64, _ = G.gemm_w4a8(q, s, p, sc, rows=rows)
    got = c if rows is None else c[:, torch.from_numpy(rows).cuda()]
    assert_gemm_matches(got, c64, f"linear M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [7, 16, 40])
def test_row_strides_and_guard_band(r4q, M):
    """x as a column slice of a wider buffer (ldx = K + 40), C inside a wider
    buffer with guard columns and rows: only C's M x N block changes."""
    N, K = 520, 1280
    pk, _, _ = _weights(r4q, N, K)
    wide = synth.activations(M, K + 40, synth.CFG_DECODE, outliers=True).cuda()
    x = wide[:, :K]
    c, full = _linear(r4q, x, pk, N, K, ldc=N + 24)
    q, s = r4q.quant_fp8(x.contiguous())
    ref = r4q.gemm_w4a8(q, s, pk, N, K)
    check_device_error(r4q)
    assert torch.equal(c, ref)
    g = full.float().cpu().numpy()
    assert np.all(g[:M, N:] == 7.0), "wrote outside columns [0, N)"
    assert np.all(g[M:, :] == 7.0), "wrote rows past M"


def test_workspace_reused_across_shapes(r4q):
    """One workspace for calls of different token counts and widths, one
    after another (and the plain GEMM on the same buffer): split-K counters
    stay at the start of every GEMM workspace and neither partials nor the
    quantization scratch reach another call's counters, so every call elects
    the right last CTA. (Counters placed after an M-sized scratch would move
    with M and be found non-zero by the next shape.)"""
    K = 2048
    shapes = [(16, 1024), (15, 1024), (40, 640), (16, 1024), (8, 384), (16, 1024)]
    packs = {N: _weights(r4q, N, K)[0] for N in {n for _, n in shapes}}
    xs = synth.activations(40, K, synth.CFG_DECODE, outliers=True).cuda()
    size = max(r4q.r4_gemm_workspace_bytes(r4q.R4_OP_LINEAR_W4A8_MXFP4, M, N, K) for M, N in shapes)
    size = max(size, max(r4q.r4_gemm_workspace_bytes(r4q.R4_OP_W4A8_MXFP4, M, N, K) for M, N in shapes))
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for M, N in shapes:
            x = xs[:M]
            c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            r4q.r4_linear_w4a8_mxfp4(x, K, packs[N], M, N, K, c, N, ws)
            q, s = r4q.quant_fp8(x)
            c2 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            r4q.r4_gemm_w4a8_mxfp4(q, s, packs[N], M, N, K, c2, N, ws)
            ref = r4q.gemm_w4a8(q, s, packs[N], N, K)
            check_device_error(r4q)
            assert torch.equal(c, ref), f"linear M={M} N={N} (pass {rep})"
            assert torch.equal(c2, ref), f"GEMM M={M} N={N} on the shared workspace (pass {rep})"
