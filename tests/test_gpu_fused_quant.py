"""GPU parity: fused quantization producers (add + Gemma RMS norm + quant,
SiluAndMul + quant) against the oracle.

The new residual is compared bit for bit. The codes and scales are integers
decided by floating point: given its scale, a code is a fixed function of the
bfloat16 value h it quantizes, and h is the one value whose rounding depends
on arithmetic order (the kernel forms the norm, and SiLU's exponential, in
fp32; the oracle in float64). So for every element the test derives the
bfloat16 values h can take -- one, or the two neighbours when the exact value
lies within 2^-20 (relative) of a bfloat16 rounding boundary -- and requires
the kernel's scale to come from a row maximum over those candidates and each
kernel code to be the oracle encoder's code of one candidate under the
kernel's own scale (same decision, same precision). Ambiguous elements must
stay rare, so the check cannot pass vacuously."""

import numpy as np
import pytest
import torch

from block_scaled_precision_token_gb300 import synth
from oracle import formats as F
from oracle import fused as U
from oracle import quant as Q
from tests.gpu_util import bf16_to_np, check_device_error, np_f32, np_u8, require_gpu

pytestmark = pytest.mark.gpu

_REL = 2.0 ** -20


@pytest.fixture(scope="module")
def r4q():
    return require_gpu()


def _randn(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def _candidates(x64):
    """bfloat16 values an fp32 computation of the exact x64 may round to."""
    lo = F.bf16_round(x64 * (1 - _REL))
    hi = F.bf16_round(x64 * (1 + _REL))
    return np.minimum(lo, hi), np.maximum(lo, hi)


def _codes_of(h, s):
    """The per-token rule's codes of bfloat16 values h under fp32 scales s
    (one correctly rounded fp32 division each, as in the oracle's quant_act)."""
    return F.e4m3_encode_rne_sat((h.astype(np.float32) / s[:, None]).astype(np.float32))


def _check_quant(q_gpu, s_gpu, h_lo, h_hi, what):
    q = np_u8(q_gpu)
    s = np_f32(s_gpu).astype(np.float32)
    amax_lo = np.max(np.minimum(np.abs(h_lo), np.abs(h_hi)), axis=1)
    amax_hi = np.max(np.maximum(np.abs(h_lo), np.abs(h_hi)), axis=1)
    s_lo = np.maximum((amax_lo.astype(np.float32) / Q.FP8_MAX).astype(np.float32), Q.MIN_SCALE)
    s_hi = np.maximum((amax_hi.astype(np.float32) / Q.FP8_MAX).astype(np.float32), Q.MIN_SCALE)
    assert np.all((s >= s_lo) & (s <= s_hi)), f"{what}: scale outside the candidates' range"
    c_lo, c_hi = _codes_of(h_lo, s), _codes_of(h_hi, s)
    ok = (q == c_lo) | (q == c_hi)
    assert ok.all(), f"{what}: {np.count_nonzero(~ok)} codes match neither candidate"
    ambiguous = np.count_nonzero(h_lo != h_hi)
    assert ambiguous <= max(2, 0.01 * h_lo.size), f"{what}: {ambiguous} of {h_lo.size} elements are rounding-ambiguous"


def _run_arq(r4q, y, res, w, eps, inplace=False):
    yd, rd, wd = y.cuda(), res.cuda().clone(), w.cuda()
    q, s, ro = r4q.add_rmsnorm_quant(yd, rd, wd, eps, residual_out=rd if inplace else None)
    check_device_error(r4q)
    return q, s, ro


@pytest.mark.parametrize("M,K", [(1, 8), (7, 128), (64, 5120), (300, 2048), (33, 4104), (5, 24576)])
def test_add_rmsnorm_quant(r4q, M, K):
    y = _randn((M, K), M * 7 + K, 1.0)
    res = _randn((M, K), M * 11 + K, 3.0)
    w = _randn((K,), K, 0.1)
    eps = 1e-6
    q, s, ro = _run_arq(r4q, y, res, w, eps)
    r, h64 = U.add_rmsnorm(y.float().numpy(), res.float().numpy(), w.float().numpy(), eps)
    assert np.array_equal(bf16_to_np(ro), r), "new residual differs"
    h_lo, h_hi = _candidates(h64)
    _check_quant(q, s, h_lo, h_hi, f"add_rmsnorm_quant M={M} K={K}")
    # one CTA per row (rows staged in shared memory), or a row over a cluster
    assert r4q.r4_last_kernel_name().startswith(("add_rmsnorm_quant_staged_kernel", "add_rmsnorm_quant_kernel"))


@pytest.mark.parametrize("M,K", [(4, 512), (400, 5120), (5, 24576)])
def test_add_rmsnorm_quant_in_place_and_zero_row(r4q, M, K):
    """residual_out = residual: one CTA per row staged in shared memory (one
    pass of the block's threads, and five, where later passes are still being
    copied in while earlier columns of the same row are written back) and a
    row spread over a cluster."""
    y = _randn((M, K), 1 + M, 1.0)
    res = _randn((M, K), 2 + M, 1.0)
    res[2] = -y[2]                                   # r = 0: minimum scale, all-zero codes
    w = _randn((K,), 3 + M, 0.1)
    q, s, ro = _run_arq(r4q, y, res, w, 1e-6, inplace=True)
    name = r4q.r4_last_kernel_name()
    assert name.startswith("add_rmsnorm_quant_kernel" if K == 24576 else "add_rmsnorm_quant_staged_kernel"), name
    r, h64 = U.add_rmsnorm(y.float().numpy(), res.float().numpy(), w.float().numpy(), 1e-6)
    assert np.array_equal(bf16_to_np(ro), r)
    assert np.all(np_u8(q)[2] == 0) and np_f32(s)[2] == Q.MIN_SCALE
    h_lo, h_hi = _candidates(h64)
    _check_quant(q, s, h_lo, h_hi, "in-place")


def test_add_rmsnorm_quant_prefill_rows_sampled(r4q):
    """The full prefill hidden shape, M=8192 x K=5120, checked on sampled rows."""
    M, K = 8192, 5120
    y = _randn((M, K), 21, 1.0)
    res = _randn((M, K), 22, 2.0)
    w = _randn((K,), 23, 0.1)
    q, s, ro = _run_arq(r4q, y, res, w, 1e-6)
    rows = synth.sample_indices(M, 96, 24).numpy()
    r, h64 = U.add_rmsnorm(y[rows].float().numpy(), res[rows].float().numpy(), w.float().numpy(), 1e-6)
    assert np.array_equal(bf16_to_np(ro)[rows], r)
    h_lo, h_hi = _candidates(h64)
    rt = torch.from_numpy(rows).cuda()
    _check_quant(q[rt], s[rt], h_lo, h_hi, "prefill sampled rows")


@pytest.mark.parametrize("M,N", [(1, 8), (6, 17408), (64, 2048), (257, 1024), (3, 24576),
                                 (160, 17408), (153, 24576),    # 512-thread blocks
                                 (305, 2048), (333, 17408), (401, 24576)])   # more rows than SMs
def test_silu_mul_quant(r4q, M, N):
    g = _randn((M, N), M + N, 3.0)
    u = _randn((M, N), M + 2 * N, 1.0)
    gu = torch.cat([g, u], dim=1)
    q, s = r4q.silu_mul_quant(gu.cuda())
    check_device_error(r4q)
    # a = bf16(silu(g)) is the value whose rounding the fp32 exponential may
    # move; h = bf16(a * u) is then a single rounding of an exact product.
    g64, u64 = g.double().numpy(), u.double().numpy()
    a64 = g64 / (1.0 + np.exp(-g64))
    a_lo, a_hi = _candidates(a64)
    h1, h2 = F.bf16_round(a_lo * u64), F.bf16_round(a_hi * u64)
    _check_quant(q, s, np.minimum(h1, h2), np.maximum(h1, h2), f"silu_mul_quant M={M} N={N}")
    # the oracle's own (single-valued) result is one of the accepted ones
    qo, so, _, _ = U.silu_mul_quant(gu.float().numpy())
    assert np.mean(np_u8(q) == qo) > 0.999
    # a row per CTA (the row staged in shared memory by bulk copies) from one
    # row per SM up; shorter batches may spread a row over a cluster
    name = r4q.r4_last_kernel_name()
    if M >= torch.cuda.get_device_properties(0).multi_processor_count:
        assert name.startswith("silu_mul_quant_staged_kernel"), name
    else:
        assert name.startswith(("silu_mul_quant_kernel", "silu_mul_quant_staged_kernel")), name


@pytest.mark.parametrize("C", [1, 2, 4, 8])
@pytest.mark.parametrize("M,K", [(3, 5120), (2, 1000), (5, 8), (4, 17408)])
def test_row_split(r4q, C, M, K):
    """Rows spread over C CTAs of a cluster (partial sums of squares and
    maxima combined across the cluster) give the same accepted results."""
    y = _randn((M, K), M * 13 + K + C, 1.0)
    res = _randn((M, K), M * 17 + K + C, 2.0)
    w = _randn((K,), K + C, 0.1)
    g = _randn((M, K), M * 19 + K + C, 3.0)
    u = _randn((M, K), M * 23 + K + C, 1.0)
    r4q.r4_set_option(11, C)
    try:
        q, s, ro = _run_arq(r4q, y, res, w, 1e-6)
        q2, s2 = r4q.silu_mul_quant(torch.cat([g, u], dim=1).cuda())
        check_device_error(r4q)
    finally:
        r4q.r4_set_option(11, 0)
    r, h64 = U.add_rmsnorm(y.float().numpy(), res.float().numpy(), w.float().numpy(), 1e-6)
    assert np.array_equal(bf16_to_np(ro), r)
    h_lo, h_hi = _candidates(h64)
    _check_quant(q, s, h_lo, h_hi, f"add_rmsnorm_quant C={C} M={M} K={K}")
    g64, u64 = g.double().numpy(), u.double().numpy()
    a_lo, a_hi = _candidates(g64 / (1.0 + np.exp(-g64)))
    h1, h2 = F.bf16_round(a_lo * u64), F.bf16_round(a_hi * u64)
    _check_quant(q2, s2, np.minimum(h1, h2), np.maximum(h1, h2), f"silu_mul_quant C={C} M={M} N={K}")


@pytest.mark.parametrize("T", [64, 128])
@pytest.mark.parametrize("M,K", [(300, 5120), (3, 24576), (4, 1000)])
def test_block_size_cap(r4q, T, M, K):
    """Option 13 caps the threads per CTA of both producers."""
    y = _randn((M, K), M * 29 + K + T, 1.0)
    res = _randn((M, K), M * 37 + K + T, 2.0)
    w = _randn((K,), K + T, 0.1)
    g = _randn((M, K), M * 41 + K + T, 3.0)
    u = _randn((M, K), M * 43 + K + T, 1.0)
    r4q.r4_set_option(13, T)
    try:
        q, s, ro = _run_arq(r4q, y, res, w, 1e-6)
        q2, s2 = r4q.silu_mul_quant(torch.cat([g, u], dim=1).cuda())
        check_device_error(r4q)
    finally:
        r4q.r4_set_option(13, 0)
    r, h64 = U.add_rmsnorm(y.float().numpy(), res.float().numpy(), w.float().numpy(), 1e-6)
    assert np.array_equal(bf16_to_np(ro), r)
    h_lo, h_hi = _candidates(h64)
    _check_quant(q, s, h_lo, h_hi, f"add_rmsnorm_quant T={T} M={M} K={K}")
    g64, u64 = g.double().numpy(), u.double().numpy()
    a_lo, a_hi = _candidates(g64 / (1.0 + np.exp(-g64)))
    h1, h2 = F.bf16_round(a_lo * u64), F.bf16_round(a_hi * u64)
    _check_quant(q2, s2, np.minimum(h1, h2), np.maximum(h1, h2), f"silu_mul_quant T={T} M={M} N={K}")


def test_fused_quant_argument_checks(r4q):
    y = torch.zeros((2, 12), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((12,), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((2, 12), dtype=torch.uint8, device="cuda")
    s = torch.zeros((2,), dtype=torch.float32, device="cuda")
    with pytest.raises(r4q.R4Error) as ei:
        r4q.r4_add_rmsnorm_quant_fp8(y, y, w, 1e-6, 2, 12, y, q, s)
    assert ei.value.status == r4q.R4_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(r4q.R4Error) as ei:
        r4q.r4_add_rmsnorm_quant_fp8(y, y, w, -1.0, 2, 8, y, q, s)
    assert ei.value.status == r4q.R4_ERR_INVALID_ARG
    gu = torch.zeros((2, 24), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(r4q.R4Error) as ei:
        r4q.r4_silu_mul_quant_fp8(gu, 2, 12, q, s)
    assert ei.value.status == r4q.R4_ERR_UNSUPPORTED_SHAPE
