"""GPU parity: skinny bf16 NT GEMM (cluster split-K, DSMEM reduction)."""

import numpy as np
import pytest
import torch

from block_scaled_precision_token_gb300 import synth
from oracle import gemm as G
from tests.gpu_util import assert_gemm_matches, bf16_to_np, check_device_error, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def r4q():
    return require_gpu()


@pytest.mark.parametrize("M", synth.SKINNY_M)
@pytest.mark.parametrize("N,K", synth.SKINNY_NK)
def test_workload_shapes(r4q, M, N, K):
    x = synth.activations(M, K, synth.CFG_SKINNY)
    w = synth.weights_bf16(N, K, synth.CFG_SKINNY)
    c = r4q.gemm_bf16_skinny(x.cuda(), w.cuda())
    check_device_error(r4q)
    c64, cb = G.gemm_bf16(x.float().numpy(), w.float().numpy())
    assert_gemm_matches(c, c64, f"M={M} N={N} K={K}")
    assert np.mean(bf16_to_np(c) == cb) > 0.95


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (7, 100, 512), (33, 48, 5120), (64, 1280, 5120),
                                   (13, 17, 2304), (64, 256, 16384)])
def test_ragged_shapes(r4q, M, N, K):
    x = synth.activations(M, K, synth.CFG_SKINNY, seed=9)
    w = synth.weights_bf16(N, K, synth.CFG_SKINNY, seed=10)
    out = torch.full((M, N + 8), 5.0, dtype=torch.bfloat16, device="cuda")
    c = r4q.gemm_bf16_skinny(x.cuda(), w.cuda(), out=out[:, :N])
    check_device_error(r4q)
    c64, _ = G.gemm_bf16(x.float().numpy(), w.float().numpy())
    assert_gemm_matches(c, c64, f"M={M} N={N} K={K}")
    assert torch.all(out[:, N:] == 5.0)
