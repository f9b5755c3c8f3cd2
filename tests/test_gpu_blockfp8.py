"""GPU parity: block-FP8 W8A8 GEMM (tcgen05 kind::f8f6f4 + register promotion)."""

import numpy as np
import pytest
import torch

from block_scaled_precision_token_gb300 import synth
from oracle import gemm as G
from oracle import quant as Q
from tests.gpu_util import assert_gemm_matches, check_device_error, random_e4m3_codes, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def r4q():
    m = require_gpu()
    yield m
    m.r4_set_option(3, 0)
    m.r4_set_option(8, 0)


def _run(r4q, q_np, As_np, w_np, Ws_np, N, K):
    q = torch.from_numpy(q_np).cuda()
    As = torch.from_numpy(np.ascontiguousarray(As_np, np.float32)).cuda()
    pk = r4q.prepack_blockfp8(torch.from_numpy(w_np).cuda(), torch.from_numpy(np.asarray(Ws_np, np.float32)).cuda(),
                              N, K)
    c = r4q.gemm_blockfp8(q, As, pk, N, K)
    check_device_error(r4q)
    return c


def _inputs(M, N, K, seed=0):
    x = synth.activations(M, K, synth.CFG_BLOCKFP8, outliers=False, seed=1000 + synth.CFG_BLOCKFP8 + seed)
    q, As = Q.quant_act(x.float().numpy(), group=128)
    w = synth.weights_fp32(N, K, synth.CFG_BLOCKFP8)
    wq, Ws = Q.quant_blockfp8_w(w.numpy())
    return q, As, wq, Ws


def test_scale_placement_one_hot(r4q):
    M, N, K = 8, 256, 384
    q = np.zeros((M, K), np.uint8)
    w = np.zeros((N, K), np.uint8)
    q[:, 130] = 0x38
    q[:, 300] = 0x40
    w[200, 130] = 0x38
    w[7, 300] = 0x30
    As = np.arange(1, 1 + M * 3, dtype=np.float32).reshape(M, 3)
    Ws = np.array([[13, 17, 19], [23, 29, 31]], np.float32)
    c = _run(r4q, q, As, w, Ws, N, K)
    c64, _ = G.gemm_blockfp8(q, As, w, Ws)
    assert_gemm_matches(c, c64, "one-hot")


@pytest.mark.parametrize("M", synth.BLOCKFP8_M)
@pytest.mark.parametrize("N,K", synth.BLOCKFP8_NK)
def test_workload_shapes(r4q, M, N, K):
    q, As, wq, Ws = _inputs(M, N, K)
    c = _run(r4q, q, As, wq, Ws, N, K)
    rows = None if M <= 64 else synth.sample_indices(N, 256, 5).numpy()
    c64, _ = G.gemm_blockfp8(q, As, wq, Ws, rows=rows)
    got = c if rows is None else c[:, torch.from_numpy(rows).cuda()]
    assert_gemm_matches(got, c64, f"M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [45, 200])
@pytest.mark.parametrize("splits", [1, 2, 5, 16])
def test_forced_splits_ragged_m(r4q, splits, M):
    """32-token tiles (M=45) and 128-token tiles (M=200, token-major
    accumulator), each with a ragged last tile, at forced K splits."""
    N, K = 384, 2048
    q = random_e4m3_codes((M, K), seed=3)
    As = np.random.default_rng(4).uniform(1e-3, 1e-2, (M, K // 128)).astype(np.float32)
    w = random_e4m3_codes((N, K), seed=5)
    Ws = np.random.default_rng(6).uniform(1e-4, 1e-3, (N // 128, K // 128)).astype(np.float32)
    r4q.r4_set_option(3, splits)
    try:
        c = _run(r4q, q, As, w, Ws, N, K)
        c2 = _run(r4q, q, As, w, Ws, N, K)
    finally:
        r4q.r4_set_option(3, 0)
    c64, _ = G.gemm_blockfp8(q, As, w, Ws)
    assert_gemm_matches(c, c64, f"splits={splits}")
    assert torch.equal(c, c2)


# the 128-token tile's variants: (weight rows, kernel)
VARIANTS_128 = [(128, "blockfp8_f8f6f4_kernel<128>"), (256, "blockfp8_f8f6f4_kernel<128, 256>")]


@pytest.mark.parametrize("M,N,K", [(200, 768, 2048), (300, 1024, 1024), (129, 2048, 512), (1000, 512, 4096)])
@pytest.mark.parametrize("splits", [1, 3])
def test_weight_tile_widths(r4q, M, N, K, splits):
    """The 128-token tile with 128 and with 256 weight rows (two weight scale
    blocks side by side, one N = 256 MMA per K step, two 256-column
    accumulators): both give the oracle's result and the same bits -- every
    output's K-block sums and promotion steps are the same -- unsplit and
    with K split (fp32 partials per 128-row half), with a ragged last token
    tile and several units per CTA."""
    q = random_e4m3_codes((M, K), seed=M + K)
    As = np.random.default_rng(M + 21).uniform(1e-3, 1e-2, (M, K // 128)).astype(np.float32)
    w = random_e4m3_codes((N, K), seed=N + 22)
    Ws = np.random.default_rng(N + 23).uniform(1e-4, 1e-3, (N // 128, K // 128)).astype(np.float32)
    outs = {}
    r4q.r4_set_option(3, splits)
    try:
        for bn, name in VARIANTS_128:
            r4q.r4_set_option(8, bn)
            outs[name] = _run(r4q, q, As, w, Ws, N, K)
            assert r4q.r4_last_kernel_name() == name
    finally:
        r4q.r4_set_option(8, 0)
        r4q.r4_set_option(3, 0)
    c64, _ = G.gemm_blockfp8(q, As, w, Ws)
    for name, c in outs.items():
        assert_gemm_matches(c, c64, f"{name} splits={splits}")
    first = outs[VARIANTS_128[0][1]]
    for name, c in outs.items():
        assert torch.equal(c, first), name


def test_end_to_end_group_quant(r4q):
    M, N, K = 64, 2048, 6144
    x = synth.activations(M, K, synth.CFG_BLOCKFP8)
    w = synth.weights_fp32(N, K, synth.CFG_BLOCKFP8)
    wq, Ws = Q.quant_blockfp8_w(w.numpy())
    qg, Asg = r4q.quant_fp8(x.cuda(), group=128)
    pk = r4q.prepack_blockfp8(torch.from_numpy(wq).cuda(), torch.from_numpy(Ws).cuda(), N, K)
    c = r4q.gemm_blockfp8(qg, Asg, pk, N, K)
    check_device_error(r4q)
    q, As = Q.quant_act(x.float().numpy(), group=128)
    c64, _ = G.gemm_blockfp8(q, As, wq, Ws)
    assert_gemm_matches(c, c64, "end-to-end")


@pytest.mark.parametrize("M,N,K", [(1, 384, 1024), (13, 51200, 2048), (16, 256, 640), (17, 1024, 4096),
                                   (33, 768, 1152), (100, 2048, 1024), (129, 384, 512), (300, 8192, 1024)])
def test_token_tiles_ragged(r4q, M, N, K):
    """Every token tile (16/32/64/128) with a ragged last tile; the larger
    cases give each CTA several units, so the K-block slots wrap the scale
    ring and the tensor-memory accumulator buffers many times."""
    q = random_e4m3_codes((M, K), seed=M)
    As = np.random.default_rng(M + 1).uniform(1e-3, 1e-2, (M, K // 128)).astype(np.float32)
    w = random_e4m3_codes((N, K), seed=M + 2)
    Ws = np.random.default_rng(M + 3).uniform(1e-4, 1e-3, (N // 128, K // 128)).astype(np.float32)
    c = _run(r4q, q, As, w, Ws, N, K)
    rows = None if N <= 2048 else synth.sample_indices(N, 384, M).numpy()
    c64, _ = G.gemm_blockfp8(q, As, w, Ws, rows=rows)
    got = c if rows is None else c[:, torch.from_numpy(rows).cuda()]
    assert_gemm_matches(got, c64, f"M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K,pad", [(300, 1024, 1024, 8), (300, 1024, 1024, 1), (64, 6144, 2048, 24),
                                       (45, 384, 2048, 3), (200, 768, 512, 0)])
def test_output_row_stride_guard_band(r4q, M, N, K, pad):
    """C inside a larger buffer: a row stride that is a 16-byte multiple
    (the tiles leave through TMA tensor stores) and one that is not (plain
    stores), ragged token tiles (the tensor store clips rows past M), more
    than one unit per CTA. The K split is forced to 1 (the unsplit tiles
    are the ones stored from shared memory). Only the M x N block changes."""
    q = random_e4m3_codes((M, K), seed=M + pad)
    As = np.random.default_rng(M + 11).uniform(1e-3, 1e-2, (M, K // 128)).astype(np.float32)
    w = random_e4m3_codes((N, K), seed=N + pad)
    Ws = np.random.default_rng(N + 13).uniform(1e-4, 1e-3, (N // 128, K // 128)).astype(np.float32)
    pk = r4q.prepack_blockfp8(torch.from_numpy(w).cuda(), torch.from_numpy(Ws).cuda(), N, K)
    ldc = N + pad
    full = torch.full((M + 3, ldc), 7.0, dtype=torch.bfloat16, device="cuda")
    r4q.r4_set_option(3, 1)
    try:
        ws = r4q.workspace(r4q.R4_OP_BLOCKFP8, M, N, K)
        r4q.r4_gemm_blockfp8(torch.from_numpy(q).cuda(), torch.from_numpy(As).cuda(), pk, M, N, K, full, ldc, ws)
        check_device_error(r4q)
    finally:
        r4q.r4_set_option(3, 0)
    rows = None if N <= 2048 else synth.sample_indices(N, 384, M).numpy()
    c64, _ = G.gemm_blockfp8(q, As, w, Ws, rows=rows)
    c = full[:M, :N]
    got = c if rows is None else c[:, torch.from_numpy(rows).cuda()]
    assert_gemm_matches(got, c64, f"M={M} N={N} K={K} ldc={ldc}")
    g = full.float().cpu().numpy()
    assert np.all(g[:M, N:] == 7.0), "kernel wrote outside columns [0, N)"
    assert np.all(g[M:, :] == 7.0), "kernel wrote rows past M"
