"""GPU parity: r4_linear_w4a8_mxfp4, per-token quantization + W4A8 GEMM from
bf16 activations. For M <= 16 the quantization runs inside the GEMM kernel
(its producer warps write the e4m3 activation tiles); the result must equal
the two-launch path (the quantization kernel, then r4_gemm_w4a8_mxfp4) bit
for bit, and the oracle's quantize-then-GEMM within the GEMM tolerance."""

import numpy as np
import pytest
import torch

from block_scaled_precision_token_gb300 import synth
from oracle import gemm as G
from oracle import quant as Q
from tests.gpu_util import assert_gemm_matches, check_device_error, require_gpu

pytestmark = pytest.mark.gpu

FUSE = 17   # option key: quantize inside the 16-token GEMM tile (1) or launch the quantizer (0)


@pytest.fixture(scope="module")
def r4q():
    m = require_gpu()
    yield m
    m.r4_set_option(FUSE, 0)
    m.r4_set_option(10, 0)
    m.r4_set_option(1, 0)


def _weights(r4q, N, K, seed=0):
    w = synth.weights_fp32(N, K, synth.CFG_DECODE)
    if seed:
        w = w * (1.0 + 0.25 * torch.from_numpy(np.random.default_rng(seed).standard_normal(w.shape)).float())
    p, sc = Q.quant_mxfp4_ocp(w.numpy())
    pk = r4q.prepack_mxfp4(torch.from_numpy(p).cuda(), torch.from_numpy(sc).cuda(), N, K)
    return pk, p, sc


def _linear(r4q, x, pk, N, K, fuse, ldc=None):
    """x: bf16 [M, >= K] on the GPU (row stride x.stride(0))."""
    M = x.shape[0]
    r4q.r4_set_option(FUSE, fuse)
    try:
        full = None
        out = None
        if ldc is not None:
            full = torch.full((M + 2, ldc), 7.0, dtype=torch.bfloat16, device="cuda")
            out = full[:M, :N]
        ws = r4q.workspace(r4q.R4_OP_LINEAR_W4A8_MXFP4, M, N, K)
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda") if out is None else out
        r4q.r4_linear_w4a8_mxfp4(x, x.stride(0), pk, M, N, K, c, c.stride(0), ws)
        check_device_error(r4q)
    finally:
        r4q.r4_set_option(FUSE, 0)
    return c, full


@pytest.mark.parametrize("N,K", [(384, 1024), (300, 416), (2048, 5120), (5120, 17408), (34816, 5120)])
@pytest.mark.parametrize("M", [1, 6, 8, 13, 16])
def test_fused_equals_two_launches(r4q, M, N, K):
    """The 16-token tile quantizing its own activations (token rows past M
    and K past the last column zero-filled, a partial last K block at
    K = 416, split-K schedules on 5120 x 17408) gives exactly the bits of
    quantizing first."""
    pk, _, _ = _weights(r4q, N, K)
    x = synth.activations(M, K, synth.CFG_DECODE, outliers=True).cuda()
    fused, _ = _linear(r4q, x, pk, N, K, fuse=1)
    two, _ = _linear(r4q, x, pk, N, K, fuse=0)
    q, s = r4q.quant_fp8(x)
    ref = r4q.gemm_w4a8(q, s, pk, N, K)
    check_device_error(r4q)
    assert torch.equal(two, ref), "two-launch path differs from quant + GEMM"
    assert torch.equal(fused, ref), "fused quantization differs from quant + GEMM"


@pytest.mark.parametrize("M,N,K", [(6, 640, 1792), (16, 2048, 5120), (11, 5120, 17408)])
def test_fused_against_oracle(r4q, M, N, K):
    pk, p, sc = _weights(r4q, N, K, seed=M)
    x = synth.activations(M, K, synth.CFG_DECODE, outliers=True)
    c, _ = _linear(r4q, x.cuda(), pk, N, K, fuse=1)
    q, s = Q.quant_act(x.float().numpy())
    rows = None if N <= 2048 else synth.sample_indices(N, 384, M).numpy()
    c64, _ = G.gemm_w4a8(q, s, p, sc, rows=rows)
    got = c if rows is None else c[:, torch.from_numpy(rows).cuda()]
    assert_gemm_matches(got, c64, f"fused M={M} N={N} K={K}")


@pytest.mark.parametrize("fuse", [1, 0])
@pytest.mark.parametrize("M", [7, 16, 40])
def test_row_strides_and_guard_band(r4q, fuse, M):
    """x as a column slice of a wider buffer (ldx = K + 40), C inside a wider
    buffer with guard columns and rows: only C's M x N block changes. M = 40
    takes the two-launch path whatever the option."""
    N, K = 520, 1280
    pk, _, _ = _weights(r4q, N, K)
    wide = synth.activations(M, K + 40, synth.CFG_DECODE, outliers=True).cuda()
    x = wide[:, :K]
    c, full = _linear(r4q, x, pk, N, K, fuse=fuse, ldc=N + 24)
    q, s = r4q.quant_fp8(x.contiguous())
    ref = r4q.gemm_w4a8(q, s, pk, N, K)
    check_device_error(r4q)
    assert torch.equal(c, ref)
    g = full.float().cpu().numpy()
    assert np.all(g[:M, N:] == 7.0), "wrote outside columns [0, N)"
    assert np.all(g[M:, :] == 7.0), "wrote rows past M"


@pytest.mark.parametrize("M", [17, 32, 64])
def test_two_launch_path_above_16_tokens(r4q, M):
    N, K = 2048, 5120
    pk, _, _ = _weights(r4q, N, K)
    x = synth.activations(M, K, synth.CFG_DECODE, outliers=True).cuda()
    c, _ = _linear(r4q, x, pk, N, K, fuse=1)
    q, s = r4q.quant_fp8(x)
    ref = r4q.gemm_w4a8(q, s, pk, N, K)
    check_device_error(r4q)
    assert torch.equal(c, ref)


def test_special_rows(r4q):
    """Rows of zeros (scale floor), a single huge value, tiny subnormal-range
    values and negative zero: the fused quantizer takes the quantization
    kernel's decisions exactly."""
    M, N, K = 9, 384, 2048
    pk, _, _ = _weights(r4q, N, K)
    x = synth.activations(M, K, synth.CFG_DECODE, outliers=False).clone()
    x[0] = 0.0
    x[1, 17] = 3.0e4
    x[2] = x[2] * 1e-30
    x[3] = -0.0
    x[4, :] = 1.0
    fused, _ = _linear(r4q, x.cuda(), pk, N, K, fuse=1)
    q, s = r4q.quant_fp8(x.cuda())
    ref = r4q.gemm_w4a8(q, s, pk, N, K)
    check_device_error(r4q)
    assert torch.equal(fused, ref)


def test_workspace_reused_across_shapes(r4q):
    """One workspace for calls of different token counts and widths, one
    after another (fused 16 and 15 tokens, the two-launch path at 40 tokens,
    and the plain GEMM on the same buffer): split-K counters stay at the
    start of every GEMM workspace and no call's partials or quantization
    scratch reach another's counters, so every call elects the right last
    CTA. (Counters placed after an M-sized scratch would move with M and
    be found non-zero by the next shape.)"""
    K = 2048
    shapes = [(16, 1024), (15, 1024), (40, 640), (16, 1024), (8, 384), (16, 1024)]
    packs = {N: _weights(r4q, N, K)[0] for N in {n for _, n in shapes}}
    xs = synth.activations(40, K, synth.CFG_DECODE, outliers=True).cuda()
    size = max(r4q.r4_gemm_workspace_bytes(r4q.R4_OP_LINEAR_W4A8_MXFP4, M, N, K) for M, N in shapes)
    size = max(size, max(r4q.r4_gemm_workspace_bytes(r4q.R4_OP_W4A8_MXFP4, M, N, K) for M, N in shapes))
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    r4q.r4_set_option(FUSE, 1)
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
    r4q.r4_set_option(FUSE, 0)
