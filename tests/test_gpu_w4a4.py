"""GPU parity: the W4A4 variant -- MXFP4 activation quantization and the
MXFP4 x MXFP4 GEMM on tcgen05 kind::mxf4 -- against the oracle."""

import numpy as np
import pytest
import torch

from block_scaled_precision_token_gb300 import synth
from oracle import formats as F
from oracle import gemm as G
from oracle import quant as Q
from tests.gpu_util import assert_gemm_matches, bf16_to_np, check_device_error, np_u8, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def r4q():
    m = require_gpu()
    yield m
    m.r4_set_option(1, 0)
    m.r4_set_option(2, 0)
    m.r4_set_option(6, 1)


def act_scale_atoms(scale, M, K):
    """Test-side permutation of scale codes [M, K/32] into the atom layout the
    GEMM reads: atoms K-block-major, atom (a, kb) at (kb * A + a) * 512; its
    byte 16 r0 + 4 r1 + j = token 128 a + 32 r1 + r0, 32-K block 4 kb + j;
    padding code 127."""
    A = -(-M // 256) * 2
    KB = -(-K // 128)
    full = np.full((A * 128, KB * 4), 127, np.uint8)
    full[:M, :K // 32] = scale
    # [a][r1][r0][kb][j] -> [kb][a][r0][r1][j]
    return np.ascontiguousarray(full.reshape(A, 4, 32, KB, 4).transpose(3, 0, 2, 1, 4)).reshape(-1)


def act_scale_codes(atoms, M, K):
    """Inverse of act_scale_atoms: (scale [M, K/32], padding all 127)."""
    A = -(-M // 256) * 2
    KB = -(-K // 128)
    # [kb][a][r0][r1][j] -> [a][r1][r0][kb][j]
    full = np.asarray(atoms, np.uint8).reshape(KB, A, 32, 4, 4).transpose(1, 3, 2, 0, 4).reshape(A * 128, KB * 4)
    pad_ok = bool(np.all(full[M:] == 127) and np.all(full[:, K // 32:] == 127))
    return full[:M, :K // 32], pad_ok


def test_atom_helpers_round_trip():
    rng = np.random.default_rng(0)
    sc = rng.integers(0, 255, (37, 416 // 32), dtype=np.uint8)
    back, pad_ok = act_scale_codes(act_scale_atoms(sc, 37, 416), 37, 416)
    assert pad_ok and np.array_equal(back, sc)


def _quant_check(r4q, x, what):
    M, K = x.shape
    q, sc = r4q.quant_mxfp4(x.cuda())
    check_device_error(r4q)
    q_ref, sc_ref = Q.quant_act_mxfp4(x.float().numpy())
    codes, pad_ok = act_scale_codes(np_u8(sc), M, K)
    assert pad_ok, f"{what}: scale padding is not code 127"
    assert np.array_equal(codes, sc_ref), f"{what}: scale codes differ"
    assert np.array_equal(np_u8(q), q_ref), f"{what}: e2m1 codes differ"


@pytest.mark.parametrize("M,K", [(8, 2048), (37, 416), (300, 5120), (6, 17408), (64, 5120), (2048, 6144)])
def test_quant_mxfp4_bit_exact(r4q, M, K):
    x = synth.activations(M, K, synth.CFG_DECODE, outliers=True)
    _quant_check(r4q, x, f"M={M} K={K}")


def test_quant_mxfp4_special_rows(r4q):
    """Zero blocks (code 127), negative zeros and negatives that round to zero
    (code 8), saturation at +-6, ties, tiny and huge magnitudes (scale codes
    near both clamps), and a strided row."""
    K = 512
    rows = []
    rows.append(np.zeros(K))
    r = np.zeros(K); r[::2] = -0.0; r[1::2] = -1e-30; rows.append(r)
    r = np.linspace(-6.5, 6.5, K); rows.append(r)                       # within one block: saturation
    r = np.tile([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 4.0], K // 8); rows.append(r)   # e2m1 ties (X = 0)
    r = np.full(K, 3e-38); r[5] = 1e-39; rows.append(r)                 # tiny: X clamped at -127
    r = np.full(K, 3e38); r[::3] = -1e38; rows.append(r)                # huge
    r = synth.activations(1, K, synth.CFG_TINY).float().numpy()[0] * 2.0 ** -100; rows.append(r)
    x = torch.tensor(np.stack(rows), dtype=torch.float32).to(torch.bfloat16)
    _quant_check(r4q, x, "special rows")
    # a row stride larger than K
    xs = synth.activations(16, 640, synth.CFG_TINY, outliers=False)
    q, sc = r4q.quant_mxfp4(xs.cuda()[:, :512])
    check_device_error(r4q)
    q_ref, sc_ref = Q.quant_act_mxfp4(xs[:, :512].float().numpy())
    codes, _ = act_scale_codes(np_u8(sc), 16, 512)
    assert np.array_equal(np_u8(q), q_ref) and np.array_equal(codes, sc_ref)


def _run(r4q, xq, xsc, M, K, wp, wsc, N, ldc=None):
    q = torch.from_numpy(np.ascontiguousarray(xq)).cuda()
    sc = torch.from_numpy(act_scale_atoms(xsc, M, K)).cuda()
    pk = r4q.prepack_mxfp4(torch.from_numpy(wp).cuda(), torch.from_numpy(wsc).cuda(), N, K)
    full = out = None
    if ldc is not None:
        full = torch.full((M, ldc), 7.0, dtype=torch.bfloat16, device="cuda")
        out = full[:, :N]
    c = r4q.gemm_w4a4(q, sc, pk, N, K, out=out)
    check_device_error(r4q)
    return c, full


def _dense(M, N, K, cfg, outliers=True):
    x = synth.activations(M, K, cfg, outliers=outliers)
    xq, xsc = Q.quant_act_mxfp4(x.float().numpy())
    w = synth.weights_fp32(N, K, cfg)
    wp, wsc = Q.quant_mxfp4_ocp(w.numpy())
    return xq, xsc, wp, wsc


def test_one_hot_weights(r4q):
    """One nonzero e2m1 weight per row at a row-dependent k (odd and even) with
    a row-dependent scale: pins the weight nibble order and scale placement."""
    M, N, K = 16, 256, 256
    rng = np.random.default_rng(0)
    xq = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    xsc = rng.integers(120, 130, (M, K // 32), dtype=np.uint8)
    codes = np.zeros((N, K), np.uint8)
    wsc = np.full((N, K // 32), 127, np.uint8)
    for n in range(N):
        k = (n * 37 + n // 7) % K
        codes[n, k] = [1, 2, 3, 4, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15][n % 14]
        wsc[n, k // 32] = 118 + (n % 13)
    wp = F.pack_e2m1(codes)
    c, _ = _run(r4q, xq, xsc, M, K, wp, wsc, N)
    c64, _ = G.gemm_w4a4(xq, xsc, wp, wsc)
    assert_gemm_matches(c, c64, "one-hot weights")


@pytest.mark.parametrize("M", [48, 200, 384])
def test_one_hot_activations(r4q, M):
    """One nonzero e2m1 activation per token at a token-dependent k with a
    token-dependent scale, against dense weights: pins the activation nibble
    order and where every token's scale sits in tensor memory (one 64-token
    tile; 256-token tiles over both atoms of a tile; a second tile)."""
    N, K = 256, 512
    rng = np.random.default_rng(1)
    codes = np.zeros((M, K), np.uint8)
    xsc = np.full((M, K // 32), 127, np.uint8)
    for m in range(M):
        k = (m * 53 + m // 5) % K
        codes[m, k] = [1, 2, 3, 4, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15][m % 14]
        xsc[m, k // 32] = 119 + (m % 11)
    xq = F.pack_e2m1(codes)
    wp = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    wsc = rng.integers(121, 128, (N, K // 32), dtype=np.uint8)
    c, _ = _run(r4q, xq, xsc, M, K, wp, wsc, N)
    c64, _ = G.gemm_w4a4(xq, xsc, wp, wsc)
    assert_gemm_matches(c, c64, f"one-hot activations M={M}")


def test_tiny_and_end_to_end(r4q):
    """x -> GPU MXFP4 quant -> GPU W4A4 GEMM equals oracle quant -> oracle GEMM
    (the quantizer is bit-exact, so the GEMM tolerance applies unchanged)."""
    M, N, K = synth.TINY["M"], synth.TINY["N"], synth.TINY["K"]
    x = synth.activations(M, K, synth.CFG_TINY)
    w = synth.weights_fp32(N, K, synth.CFG_TINY)
    wp, wsc = Q.quant_mxfp4_ocp(w.numpy())
    q, sc = r4q.quant_mxfp4(x.cuda())
    pk = r4q.prepack_mxfp4(torch.from_numpy(wp).cuda(), torch.from_numpy(wsc).cuda(), N, K)
    c = r4q.gemm_w4a4(q, sc, pk, N, K)
    check_device_error(r4q)
    xq, xsc = Q.quant_act_mxfp4(x.float().numpy())
    c64, cb = G.gemm_w4a4(xq, xsc, wp, wsc, exact_check=True)
    assert_gemm_matches(c, c64, "tiny end-to-end")
    assert np.mean(bf16_to_np(c) == cb) > 0.9
    # the pages' error measure against the product with unquantized
    # activations (they report 0.1119 for their W4A4 path, 0.0265 for W4A8)
    ref = x.float().numpy().astype(np.float64) @ Q.dequant_mxfp4(wp, wsc, K).T
    assert G.rel_frobenius(bf16_to_np(c), ref) < 0.3


def test_ragged_shapes_and_guard_band(r4q):
    M, N, K = 37, 300, 416
    xq, xsc, wp, wsc = _dense(M, N, K, synth.CFG_DECODE)
    c, full = _run(r4q, xq, xsc, M, K, wp, wsc, N, ldc=320)
    c64, _ = G.gemm_w4a4(xq, xsc, wp, wsc)
    assert_gemm_matches(c, c64, "ragged")
    assert np.all(full.float().cpu().numpy()[:, N:] == 7.0), "kernel wrote outside columns [0, N)"


@pytest.mark.parametrize("bt", [0, 64, 128, 192, 256])   # 192: W4A4 falls back to its own choice
@pytest.mark.parametrize("splits,cluster", [(1, 1), (3, 1), (3, 0), (8, 0)])
def test_forced_tiles_and_splits(r4q, bt, splits, cluster):
    M, N, K = 40, 384, 1024
    if bt >= 128:
        M = 300                                   # several token tiles
    xq, xsc, wp, wsc = _dense(M, N, K, synth.CFG_DECODE)
    r4q.r4_set_option(2, bt)
    r4q.r4_set_option(1, splits)
    r4q.r4_set_option(6, cluster)
    try:
        c, _ = _run(r4q, xq, xsc, M, K, wp, wsc, N)
        c2, _ = _run(r4q, xq, xsc, M, K, wp, wsc, N)
    finally:
        r4q.r4_set_option(1, 0)
        r4q.r4_set_option(2, 0)
        r4q.r4_set_option(6, 1)
    c64, _ = G.gemm_w4a4(xq, xsc, wp, wsc)
    assert_gemm_matches(c, c64, f"bt={bt} splits={splits} cluster={cluster}")
    assert torch.equal(c, c2), "not deterministic across calls"


def _sampled_full_size(r4q, M, N, K, seed, nsample=256):
    xq = synth.uniform_bytes((M, K // 2), seed=seed).numpy()
    xsc = synth.uniform_bytes((M, K // 32), seed=seed + 4, low=118, high=126).numpy()
    wp = synth.uniform_bytes((N, K // 2), seed=seed + 1).numpy()
    wsc = synth.uniform_bytes((N, K // 32), seed=seed + 2, low=117, high=125).numpy()
    c, _ = _run(r4q, xq, xsc, M, K, wp, wsc, N)
    rows = synth.sample_indices(N, nsample, seed + 3).numpy()
    rows = np.unique(np.concatenate([rows, [0, N - 1]]))
    c64, _ = G.gemm_w4a4(xq, xsc, wp, wsc, rows=rows)
    assert_gemm_matches(c[:, torch.from_numpy(rows).cuda()], c64, f"W4A4 M={M} N={N} K={K}")


# The decode and prefill shapes of the W4A8 workloads, at full size, through
# the planner's automatic schedule.
@pytest.mark.parametrize("M", synth.DECODE_M)
@pytest.mark.parametrize("N,K", synth.DECODE_NK)
def test_decode_full_size_sampled(r4q, M, N, K):
    _sampled_full_size(r4q, M, N, K, seed=300 + M)


@pytest.mark.parametrize("M", synth.PREFILL_M)
@pytest.mark.parametrize("N,K", synth.PREFILL_NK)
def test_prefill_full_size_sampled(r4q, M, N, K):
    _sampled_full_size(r4q, M, N, K, seed=400 + M, nsample=128)
