"""GPU parity: e4m3 activation quantization and the weight quantizers must be
bit-exact against the oracle."""

import numpy as np
import pytest
import torch

from block_scaled_precision_token_gb300 import synth
from oracle import quant as Q
from tests.gpu_util import check_device_error, np_f32, np_u8, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def r4q():
    return require_gpu()


def _x(M, K, cfg, outliers, seed=None):
    return synth.activations(M, K, cfg, outliers=outliers, seed=seed)


@pytest.mark.parametrize("M,K,outliers", [
    (8, 2048, False),        # tiny W4A8 workload
    (6, 5120, True), (64, 5120, True), (64, 17408, True),   # decode shapes
    (37, 384, True),         # ragged M, short K
    (1, 8, False),           # minimum
    (3, 40000, False),       # row longer than the register-resident path
    (256, 5120, True),
])
def test_per_token_bit_exact(r4q, M, K, outliers):
    x = _x(M, K, synth.CFG_DECODE, outliers)
    q_ref, s_ref = Q.quant_act(x.float().numpy())
    q, s = r4q.quant_fp8(x.cuda())
    check_device_error(r4q)
    assert np.array_equal(np_f32(s), s_ref)
    assert np.array_equal(np_u8(q), q_ref)


@pytest.mark.parametrize("M,K", [(8, 2048), (64, 6144), (2048, 4096), (5, 128), (33, 4096 + 128)])
def test_group128_bit_exact(r4q, M, K):
    x = _x(M, K, synth.CFG_BLOCKFP8, False)
    q_ref, s_ref = Q.quant_act(x.float().numpy(), group=128)
    q, s = r4q.quant_fp8(x.cuda(), group=128)
    check_device_error(r4q)
    assert np.array_equal(np_f32(s), s_ref)
    assert np.array_equal(np_u8(q), q_ref)


@pytest.mark.parametrize("C", [1, 2, 4, 8])
@pytest.mark.parametrize("M,K,ld,group", [
    (6, 17408, 17408, None),     # decode row, even split
    (3, 1000, 1000, None),       # ragged: the last CTA holds a partial slice
    (5, 8, 8, None),             # one vector: all but the first CTA hold nothing
    (4, 2048, 2056, None),       # row stride > K
    (300, 5120, 5120, None),     # more rows than SMs
    (7, 6144, 6144, 128),        # group-128 scales, slices of whole groups
    (2, 384, 384, 128),
])
def test_row_split_bit_exact(r4q, C, M, K, ld, group):
    """Each row spread over C CTAs (a thread-block cluster that agrees on the
    per-token maximum): identical codes and scales to the oracle for every C."""
    xb = _x(M, ld, synth.CFG_DECODE, True, seed=M * 1009 + K + C)
    q_ref, s_ref = Q.quant_act(xb[:, :K].float().numpy(), **({} if group is None else {"group": group}))
    r4q.r4_set_option(11, C)
    try:
        q, s = r4q.quant_fp8(xb.cuda()[:, :K], group=group)
        check_device_error(r4q)
    finally:
        r4q.r4_set_option(11, 0)
    assert np.array_equal(np_f32(s), s_ref)
    assert np.array_equal(np_u8(q), q_ref)


@pytest.mark.parametrize("T", [64, 128])
@pytest.mark.parametrize("M,K,group", [(300, 5120, None), (7, 24576, None), (33, 6144, 128), (5, 1000, None)])
def test_block_size_cap_bit_exact(r4q, T, M, K, group):
    """Option 13 caps the threads per CTA (more vectors per thread; a row
    too long for 12 vectors per thread widens the block again)."""
    x = _x(M, K, synth.CFG_DECODE, True, seed=M * 31 + K + T)
    q_ref, s_ref = Q.quant_act(x.float().numpy(), group=group)
    r4q.r4_set_option(13, T)
    try:
        q, s = r4q.quant_fp8(x.cuda(), group=group)
        check_device_error(r4q)
    finally:
        r4q.r4_set_option(13, 0)
    assert np.array_equal(np_f32(s), s_ref)
    assert np.array_equal(np_u8(q), q_ref)


def test_row_split_option_checks(r4q):
    with pytest.raises(r4q.R4Error):
        r4q.r4_set_option(11, 3)
    with pytest.raises(r4q.R4Error):
        r4q.r4_set_option(11, 16)
    with pytest.raises(r4q.R4Error):
        r4q.r4_set_option(13, 96)


def test_quotient_correctly_rounded_on_whole_domain(r4q):
    """The quantizers divide by the scale with a reciprocal and one FMA
    correction. For every finite bf16 amax, the scale the rule derives from
    it, and every bf16 x with |x| <= amax (both signs), the quotient must equal
    a correctly rounded fp32 division in its e4m3 code (~1.07e9 pairs). The
    fp32 quotients themselves may differ only where the remainder underflows
    (x within a few ulps of the fp32 normal range), far below the smallest
    e4m3 code 2^-9."""
    count = torch.zeros(4, dtype=torch.int64, device="cuda")
    ex = torch.zeros(2, dtype=torch.float32, device="cuda")
    r4q.r4_check_quotients(count, ex)
    torch.cuda.synchronize()
    check_device_error(r4q)
    n_code, n_bits, worst_bits = (int(v) for v in count[[0, 2, 3]].cpu())
    assert n_code == 0, f"{n_code} (x, s) pairs give other codes, e.g. x={ex[0].item()!r} s={ex[1].item()!r}"
    worst = np.array([worst_bits], dtype=np.uint32).view(np.float32)[0]
    assert worst < 2.0 ** -20, f"{n_bits} quotients differ, the largest {worst!r}"


def test_special_rows_and_row_stride(r4q):
    M, K, ld = 6, 1024, 1040
    base = _x(M, ld, synth.CFG_DECODE, False, seed=77).float()
    base[1] = 0.0                      # zero row -> minimum scale
    base[2] = 3.5                      # constant row -> every code 448
    base[3] = -base[3].abs()           # all negative
    base[4, :] = 0.0
    base[4, 5] = 1e-30                 # tiny amax
    xb = base.to(torch.bfloat16)
    view = xb.cuda()[:, :K]            # row stride ld > K
    q_ref, s_ref = Q.quant_act(xb[:, :K].float().numpy())
    q, s = r4q.quant_fp8(view)
    check_device_error(r4q)
    assert np.array_equal(np_f32(s), s_ref)
    assert np.array_equal(np_u8(q), q_ref)
    assert np.all(np_u8(q)[2] == 0x7E)


@pytest.mark.parametrize("N,K", [(256, 2048), (100, 96), (2048, 5120)])
def test_mxfp4_weight_quant_bit_exact(r4q, N, K):
    w = synth.weights_fp32(N, K, synth.CFG_TINY)
    w[3, :32] = 0.0                    # an all-zero block
    w[5, 40] = 10.0                    # saturating outlier block
    p_ref, s_ref = Q.quant_mxfp4_ocp(w.numpy())
    p, s = r4q.quantize_mxfp4_weight(w.cuda())
    check_device_error(r4q)
    assert np.array_equal(np_u8(s), s_ref)
    assert np.array_equal(np_u8(p), p_ref)


@pytest.mark.parametrize("N,K", [(256, 256), (2048, 6144)])
def test_blockfp8_weight_quant_bit_exact(r4q, N, K):
    w = synth.weights_fp32(N, K, synth.CFG_BLOCKFP8)
    w[128:256, 128:256] = 0.0
    c_ref, s_ref = Q.quant_blockfp8_w(w.numpy())
    c, s = r4q.quantize_blockfp8_weight(w.cuda())
    check_device_error(r4q)
    assert np.array_equal(np_f32(s), s_ref)
    assert np.array_equal(np_u8(c), c_ref)


def test_every_bf16_value_under_several_scales(r4q):
    """Each row holds every finite bfloat16 value up to its own amax, so the
    quotients x/s cover exact e4m3 ties (power-of-two scales) and land within
    a few float32 ulps of every e4m3 rounding boundary (other scales): the
    codes must still be those of the correctly rounded quotient."""
    bits = np.arange(65536, dtype=np.uint32)
    allv = (bits << 16).view(np.float32)
    allv = allv[np.isfinite(allv)]
    amaxes = [448.0, 1344.0, 0.01171875, 3.0517578e-05, 1.0078125, 57344.0, 1.0e-8]
    K = 65536
    rows = []
    for a in amaxes:
        a = float(torch.tensor(a).to(torch.bfloat16))
        v = allv[np.abs(allv) <= a]
        row = np.zeros(K, np.float32)
        row[:v.size] = v
        row[v.size] = a
        rows.append(row)
    x = torch.from_numpy(np.stack(rows)).to(torch.bfloat16)
    q_ref, s_ref = Q.quant_act(x.float().numpy())
    q, s = r4q.quant_fp8(x.cuda())
    check_device_error(r4q)
    assert np.array_equal(np_f32(s), s_ref)
    assert np.array_equal(np_u8(q), q_ref)
