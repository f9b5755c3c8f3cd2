"""GPU: the prepack kernels are exact permutations (round trip through a
test-only inverse) with the documented padding."""

import numpy as np
import pytest

from block_scaled_precision_token_gb300 import synth
from tests.gpu_util import (check_device_error, np_u8, prepack_inverse_blockfp8, prepack_inverse_mxfp4,
                            require_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def r4q():
    return require_gpu()


@pytest.mark.parametrize("N,K", [(256, 2048), (300, 416), (1, 32), (5120, 17408)])
def test_mxfp4_prepack_roundtrip(r4q, N, K):
    import torch
    codes = synth.uniform_bytes((N, K // 2), seed=11)
    scales = synth.uniform_bytes((N, K // 32), seed=12, low=100, high=140)
    packed = r4q.prepack_mxfp4(codes.cuda(), scales.cuda(), N, K)
    check_device_error(r4q)
    c, s, pad_ok = prepack_inverse_mxfp4(np_u8(packed), N, K)
    assert pad_ok
    assert np.array_equal(c, codes.numpy())
    assert np.array_equal(s, scales.numpy())


@pytest.mark.parametrize("N,K", [(128, 128), (6144, 2048), (2048, 6144)])
def test_blockfp8_prepack_roundtrip(r4q, N, K):
    import torch
    codes = synth.uniform_bytes((N, K), seed=13)
    sc = torch.rand((N // 128, K // 128), generator=torch.Generator().manual_seed(14), dtype=torch.float32)
    packed = r4q.prepack_blockfp8(codes.cuda(), sc.cuda(), N, K)
    check_device_error(r4q)
    c, s = prepack_inverse_blockfp8(np_u8(packed), N, K)
    assert np.array_equal(c, codes.numpy())
    assert np.array_equal(s, sc.numpy())
