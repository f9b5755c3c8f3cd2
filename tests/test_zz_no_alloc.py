"""GPU: the W4A8 GEMM entry point that allocates nothing.

Callers that run inside CUDA-graph capture, or that get only input/output
pointers and a stream from their host runtime, cannot allocate the split-K
workspace; r4_gemm_w4a8_mxfp4_noalloc keeps that scratch in a static device
buffer of the library. This test calls it through the C ABI twice in a row and
compares both results with r4_gemm_w4a8_mxfp4 (given a caller workspace) and
with the oracle, within the GEMM tolerance the other tests use. The file is
named to be collected last.
"""

import numpy as np
import pytest
import torch

from block_scaled_precision_token_gb300 import synth
from oracle import gemm as G
from oracle import quant as Q
from tests.gpu_util import assert_gemm_matches, bf16_to_np, check_device_error, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def r4q():
    m = require_gpu()
    yield m
    m.r4_set_option(1, 0)
    m.r4_set_option(6, 1)


def test_noalloc_matches_workspace_entry_point_twice(r4q):
    M, N, K = 8, 2048, 5120
    x = synth.activations(M, K, synth.CFG_DECODE, outliers=True)
    w = synth.weights_fp32(N, K, synth.CFG_DECODE)
    p, sc = Q.quant_mxfp4_ocp(w.numpy())
    q_np, s_np = Q.quant_act(x.float().numpy())
    q = torch.from_numpy(q_np).cuda()
    s = torch.from_numpy(s_np).cuda()
    pk = r4q.prepack_mxfp4(torch.from_numpy(p).cuda(), torch.from_numpy(sc).cuda(), N, K)
    r4q.r4_set_option(1, 4)                       # force split-K through the workspace
    r4q.r4_set_option(6, 0)                       # (not the cluster exchange) so the scratch is used
    try:
        assert r4q.r4_gemm_workspace_bytes(r4q.R4_OP_W4A8_MXFP4, M, N, K) > 0
        ref = r4q.gemm_w4a8(q, s, pk, N, K)       # existing entry point, caller workspace
        outs = []
        for _ in range(2):                        # two calls in a row share the static scratch
            c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            r4q.r4_gemm_w4a8_mxfp4_noalloc(q, s, pk, M, N, K, c, N)
            outs.append(c)
        check_device_error(r4q)
    finally:
        r4q.r4_set_option(1, 0)
        r4q.r4_set_option(6, 1)
    c64, _ = G.gemm_w4a8(q_np, s_np, p, sc)
    ref64 = bf16_to_np(ref)
    for c in outs:
        ok, ratio = G.gemm_tolerance_ok(bf16_to_np(c), ref64)
        assert ok, f"no-alloc result differs from the workspace entry point (worst error/bound {ratio:.3f})"
        assert_gemm_matches(c, c64, "no-alloc vs oracle")


def test_noalloc_rejects_schedules_beyond_its_scratch(r4q):
    M, N, K = 64, 34816, 5120
    q = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    s = torch.ones((M,), dtype=torch.float32, device="cuda")
    pk = torch.zeros(r4q.r4_prepack_mxfp4_bytes(N, K), dtype=torch.uint8, device="cuda")
    c = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    # decode tiles, K split 4 ways through the scratch (not a cluster):
    # 272 weight tiles x 4 splits of fp32 partial tiles, over 16 MiB. (Prefill
    # tiles take a split only while each CTA holds one split unit, which a
    # forced factor does not override, so they no longer reach this size.)
    r4q.r4_set_option(1, 4)
    r4q.r4_set_option(6, 0)
    try:
        assert r4q.r4_gemm_workspace_bytes(r4q.R4_OP_W4A8_MXFP4, M, N, K) > (16 << 20)
        with pytest.raises(r4q.R4Error) as ei:
            r4q.r4_gemm_w4a8_mxfp4_noalloc(q, s, pk, M, N, K, c, N)
        assert ei.value.status == r4q.R4_ERR_WORKSPACE
    finally:
        r4q.r4_set_option(1, 0)
        r4q.r4_set_option(6, 1)
    torch.cuda.synchronize()
    assert torch.count_nonzero(c) == 0            # nothing was launched
