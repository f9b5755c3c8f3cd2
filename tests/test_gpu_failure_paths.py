"""Failure detection and capture safety, on the GPU without a fault.

* A pipeline wait that can never complete (a test option withholds one TMA
  copy in the first CTA of a W4A8 or block-FP8 launch) must expire after its
  ~2 s limit, leave a device error word that r4_device_error reports, and
  leave the context usable: the next launch is correct.
* Such a launch must also leave the caller's split-K workspace as it found
  it: every arrival counter back at zero, so the next call on the SAME
  workspace elects the right last CTA and gives the oracle's result.
* Every entry point must be capturable in a CUDA graph (the library never
  allocates or synchronizes), and the graph's results must equal the eager
  ones bit for bit."""

import time

import numpy as np
import pytest
import torch

from block_scaled_precision_token_gb300 import synth
from oracle import gemm as G
from oracle import quant as Q
from tests.gpu_util import assert_gemm_matches, require_gpu

pytestmark = pytest.mark.gpu

# device error codes of the waits that can expire first here. Three bounded
# waits start together and run out together (~2 s): the MMA issuer on the
# starved pipeline stage, the epilogue on the accumulator it feeds, and the
# producer's end-of-kernel drain of that same stage (this small shape's
# slots are all issued before the producer's loop, so it reaches its drain
# at once). The first to record wins the error word.
WAIT_FULL, WAIT_EMPTY, WAIT_ACC_FULL, WAIT_ACC_EMPTY, WAIT_DRAIN = 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def r4q():
    m = require_gpu()
    yield m
    m.r4_set_option(10, 0)
    m.r4_set_option(1, 0)
    m.r4_set_option(2, 0)
    m.r4_set_option(3, 0)
    m.r4_set_option(6, 1)


def _w4a8_inputs(r4q, M, N, K):
    x = synth.activations(M, K, synth.CFG_DECODE, outliers=True)
    w = synth.weights_fp32(N, K, synth.CFG_DECODE)
    p, sc = Q.quant_mxfp4_ocp(w.numpy())
    q, s = Q.quant_act(x.float().numpy())
    pk = r4q.prepack_mxfp4(torch.from_numpy(p).cuda(), torch.from_numpy(sc).cuda(), N, K)
    return torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), pk, (q, s, p, sc)


def test_bounded_wait_expires_and_reports(r4q):
    M, N, K = 8, 512, 1024
    q, s, pk, ref = _w4a8_inputs(r4q, M, N, K)
    r4q.r4_device_error(clear=True)
    r4q.r4_set_option(10, 1)
    try:
        t0 = time.time()
        r4q.gemm_w4a8(q, s, pk, N, K)          # launch succeeds; a stage never fills
        torch.cuda.synchronize()                # returns: every wait is bounded
        elapsed = time.time() - t0
    finally:
        r4q.r4_set_option(10, 0)
    code = r4q.r4_device_error(clear=True)
    assert code in (WAIT_FULL, WAIT_ACC_FULL, WAIT_DRAIN), f"device error word {code}"
    assert 1.0 < elapsed < 30.0, f"the stalled launch took {elapsed:.1f} s"
    # the context is intact: the same call now gives the oracle's result
    c = r4q.gemm_w4a8(q, s, pk, N, K)
    torch.cuda.synchronize()
    assert r4q.r4_device_error(clear=True) == 0
    c64, _ = G.gemm_w4a8(*ref)
    assert_gemm_matches(c, c64, "after the stalled launch")


@pytest.mark.parametrize("mode,bt", [("w4a8", 256), ("w4a8", 192), ("w4a4", 256)])
def test_prefill_stall_reports_and_recovers(r4q, mode, bt):
    """The same on prefill tiles, whose roles differ from the decode ones:
    the 256-token tile's four helper warps (they wait on the accumulator and
    drain half of it), the 192-token tile's two accumulators, and the W4A4
    scale warp (it waits on every stage's full barrier and the MMA thread
    waits on its commits). CTA 0 withholds its first activation copy: every
    role's wait must expire and return, the error must be reported, and the
    next call must give the oracle's result."""
    M, N, K = 600, 1024, 1024
    x = synth.activations(M, K, synth.CFG_PREFILL)
    w = synth.weights_fp32(N, K, synth.CFG_PREFILL)
    p, sc = Q.quant_mxfp4_ocp(w.numpy())
    pk = r4q.prepack_mxfp4(torch.from_numpy(p).cuda(), torch.from_numpy(sc).cuda(), N, K)
    rows = np.unique(np.concatenate([synth.sample_indices(N, 128, 7).numpy(), [0, N - 1]]))
    if mode == "w4a8":
        q, s = Q.quant_act(x.float().numpy())
        qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
        call = lambda: r4q.gemm_w4a8(qd, sd, pk, N, K)
        exact = lambda: G.gemm_w4a8(q, s, p, sc, rows=rows)[0]
    else:
        xq, xsc = Q.quant_act_mxfp4(x.float().numpy())
        qd, qsd = r4q.quant_mxfp4(x.cuda())     # the GPU quantizer (bit-exact: test_gpu_w4a4.py)
        call = lambda: r4q.gemm_w4a4(qd, qsd, pk, N, K)
        exact = lambda: G.gemm_w4a4(xq, xsc, p, sc, rows=rows)[0]
    r4q.r4_set_option(2, bt)
    r4q.r4_set_option(1, 1)
    try:
        r4q.r4_device_error(clear=True)
        r4q.r4_set_option(10, 1)
        try:
            t0 = time.time()
            call()
            torch.cuda.synchronize()
            elapsed = time.time() - t0
        finally:
            r4q.r4_set_option(10, 0)
        code = r4q.r4_device_error(clear=True)
        assert code in (WAIT_FULL, WAIT_ACC_FULL, WAIT_DRAIN), f"device error word {code}"
        assert 1.0 < elapsed < 30.0, f"the stalled launch took {elapsed:.1f} s"
        c = call()
        torch.cuda.synchronize()
        assert r4q.r4_device_error(clear=True) == 0
    finally:
        r4q.r4_set_option(1, 0)
        r4q.r4_set_option(2, 0)
    assert_gemm_matches(c[:, torch.from_numpy(rows).cuda()], exact(), f"{mode} bt={bt} after the stalled launch")


@pytest.mark.parametrize("bn", [128, 256])
def test_blockfp8_prefill_stall_reports_and_recovers(r4q, bn):
    """The block-FP8 128-token tile (token-major accumulator, spinning
    per-K-block handshakes, TMA-stored output), with 128 and with 256 weight
    rows: CTA 0 withholds its first activation copy. The spinning waits are bounded like the others: they
    must expire and return, the error must be reported, and the next call
    must give the oracle's result. K = 512 keeps every slot within the ring,
    so the producer reaches its drain at once."""
    M, N, K = 300, 768, 512
    x = synth.activations(M, K, synth.CFG_BLOCKFP8)
    w = synth.weights_fp32(N, K, synth.CFG_BLOCKFP8)
    wq, Ws = Q.quant_blockfp8_w(w.numpy())
    q, As = Q.quant_act(x.float().numpy(), group=128)
    pk = r4q.prepack_blockfp8(torch.from_numpy(wq).cuda(), torch.from_numpy(Ws).cuda(), N, K)
    qd, Ad = torch.from_numpy(q).cuda(), torch.from_numpy(As).cuda()
    r4q.r4_set_option(3, 1)
    r4q.r4_set_option(8, bn)
    try:
        r4q.r4_device_error(clear=True)
        r4q.r4_set_option(10, 1)
        try:
            t0 = time.time()
            r4q.gemm_blockfp8(qd, Ad, pk, N, K)
            torch.cuda.synchronize()
            elapsed = time.time() - t0
        finally:
            r4q.r4_set_option(10, 0)
        code = r4q.r4_device_error(clear=True)
        assert code in (WAIT_FULL, WAIT_EMPTY, WAIT_ACC_FULL, WAIT_ACC_EMPTY, WAIT_DRAIN), f"device error word {code}"
        assert 1.0 < elapsed < 30.0, f"the stalled launch took {elapsed:.1f} s"
        c = r4q.gemm_blockfp8(qd, Ad, pk, N, K)
        torch.cuda.synchronize()
        assert r4q.r4_device_error(clear=True) == 0
        name = r4q.r4_last_kernel_name()
    finally:
        r4q.r4_set_option(3, 0)
        r4q.r4_set_option(8, 0)
    assert name == ("blockfp8_f8f6f4_kernel<128, 256>" if bn == 256 else "blockfp8_f8f6f4_kernel<128>")
    c64, _ = G.gemm_blockfp8(q, As, wq, Ws)
    assert_gemm_matches(c, c64, "block-FP8 128-token tile after the stalled launch")


@pytest.mark.parametrize("op", ["silu", "norm"])
def test_staged_producer_stall_reports_and_recovers(r4q, op):
    """The fused producers' one-CTA-per-row kernels stage each row with bulk
    copies, one mbarrier per pass of the block's threads: with option 10,
    CTA 0 arms its first pass but withholds the copies. That wait and the
    final drain must run out and return (no copy is left in flight), the
    error must be reported, and the next call must give the same bits as
    the call before the stall."""
    if op == "silu":
        M, N = 200, 2048
        gu = synth.activations(M, 2 * N, synth.CFG_PREFILL).cuda()

        def run():
            return r4q.silu_mul_quant(gu)
        name = "silu_mul_quant_staged_kernel"
    else:
        M, K = 300, 5120
        y = synth.activations(M, K, synth.CFG_PREFILL).cuda()
        res = synth.activations(M, K, synth.CFG_DECODE).cuda()
        wn = (synth.activations(1, K, synth.CFG_TINY)[0] * 0.1).to(torch.bfloat16).cuda()

        def run():
            q, s, _ = r4q.add_rmsnorm_quant(y, res, wn, 1e-6)
            return q, s
        name = "add_rmsnorm_quant_staged_kernel"
    q0, s0 = run()
    torch.cuda.synchronize()
    assert r4q.r4_last_kernel_name().startswith(name), r4q.r4_last_kernel_name()
    r4q.r4_device_error(clear=True)
    r4q.r4_set_option(10, 1)
    try:
        t0 = time.time()
        run()
        torch.cuda.synchronize()
        elapsed = time.time() - t0
    finally:
        r4q.r4_set_option(10, 0)
    code = r4q.r4_device_error(clear=True)
    assert code in (WAIT_FULL, WAIT_DRAIN), f"device error word {code}"
    assert 1.0 < elapsed < 30.0, f"the stalled launch took {elapsed:.1f} s"
    q1, s1 = run()
    torch.cuda.synchronize()
    assert r4q.r4_device_error(clear=True) == 0
    assert torch.equal(q0, q1) and torch.equal(s0, s1)


def _blockfp8_inputs(r4q, M, N, K):
    x = synth.activations(M, K, synth.CFG_BLOCKFP8)
    w = synth.weights_fp32(N, K, synth.CFG_BLOCKFP8)
    wq, Ws = Q.quant_blockfp8_w(w.numpy())
    q, As = Q.quant_act(x.float().numpy(), group=128)
    pk = r4q.prepack_blockfp8(torch.from_numpy(wq).cuda(), torch.from_numpy(Ws).cuda(), N, K)
    return torch.from_numpy(q).cuda(), torch.from_numpy(As).cuda(), pk, (q, As, wq, Ws)


@pytest.mark.parametrize("op", ["w4a8", "w4a8_stream_k", "blockfp8", "linear"])
def test_expired_wait_leaves_the_workspace_reusable(r4q, op):
    """Split-K through the caller's workspace (forced: 4 splits, no cluster
    exchange; or the stream-K schedule, where every tile is shared by eight
    CTAs of one K block each). The first CTA's stalled unit never writes its
    partial; the launch must still end with every arrival counter at zero,
    and the next call on the same workspace must match the oracle (for the
    linear call: its GEMM, whose counters lead the workspace, before the
    quantized activations)."""
    M, N, K = 8, 512, 1024
    tiles = (N // 128) * 1                       # 16-token tiles: one token tile
    if op == "linear":
        x = synth.activations(M, K, synth.CFG_DECODE, outliers=True)
        w = synth.weights_fp32(N, K, synth.CFG_DECODE)
        p, sc = Q.quant_mxfp4_ocp(w.numpy())
        qx, sx = Q.quant_act(x.float().numpy())
        pk = r4q.prepack_mxfp4(torch.from_numpy(p).cuda(), torch.from_numpy(sc).cuda(), N, K)
        xd = x.cuda()
        cd = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        r4q.r4_set_option(1, 4)
        r4q.r4_set_option(6, 0)
        opid = r4q.R4_OP_LINEAR_W4A8_MXFP4

        def call(ws):
            r4q.r4_linear_w4a8_mxfp4(xd, K, pk, M, N, K, cd, N, ws)
            return cd
        exact = lambda: G.gemm_w4a8(qx, sx, p, sc)[0]
    elif op.startswith("w4a8"):
        q, s, pk, ref = _w4a8_inputs(r4q, M, N, K)
        if op == "w4a8":
            r4q.r4_set_option(1, 4)
            r4q.r4_set_option(6, 0)
        else:
            r4q.r4_set_option(16, 2)
        opid = r4q.R4_OP_W4A8_MXFP4
        call = lambda ws: r4q.gemm_w4a8(q, s, pk, N, K, ws=ws)
        exact = lambda: G.gemm_w4a8(*ref)[0]
    else:
        q, As, pk, ref = _blockfp8_inputs(r4q, M, N, K)
        r4q.r4_set_option(3, 4)
        opid = r4q.R4_OP_BLOCKFP8
        call = lambda ws: r4q.gemm_blockfp8(q, As, pk, N, K, ws=ws)
        exact = lambda: G.gemm_blockfp8(*ref)[0]
    try:
        ws = r4q.workspace(opid, M, N, K)
        assert ws is not None, "the forced schedule should use the workspace"
        r4q.r4_device_error(clear=True)
        r4q.r4_set_option(10, 1)
        try:
            call(ws)
            torch.cuda.synchronize()
        finally:
            r4q.r4_set_option(10, 0)
        code = r4q.r4_device_error(clear=True)
        assert code in (WAIT_FULL, WAIT_ACC_FULL, WAIT_DRAIN), f"device error word {code}"
        counters = ws[:4 * tiles].view(torch.int32).cpu()   # every GEMM workspace starts with its counters
        assert torch.count_nonzero(counters) == 0, f"arrival counters left at {counters.tolist()}"
        c = call(ws)                              # the same workspace, reused
        torch.cuda.synchronize()
        assert r4q.r4_device_error(clear=True) == 0
    finally:
        r4q.r4_set_option(1, 0)
        r4q.r4_set_option(3, 0)
        r4q.r4_set_option(6, 1)
        r4q.r4_set_option(16, 0)
    assert_gemm_matches(c, exact(), f"{op} after the stalled launch, reused workspace")


def test_every_entry_point_captures_in_a_graph(r4q):
    dev = torch.device("cuda")
    M, K, N = 16, 2048, 1024
    x = synth.activations(M, K, synth.CFG_DECODE, outliers=True).to(dev)
    res = synth.activations(M, K, synth.CFG_TINY).to(dev)
    nw = (synth.activations(1, K, synth.CFG_TINY)[0] * 0.1).to(torch.bfloat16).to(dev)
    w = synth.weights_fp32(N, K, synth.CFG_DECODE).to(dev)
    p, sc = r4q.quantize_mxfp4_weight(w)
    pk = r4q.prepack_mxfp4(p, sc, N, K)
    wq, Ws = r4q.quantize_blockfp8_weight(w)
    pk8 = r4q.prepack_blockfp8(wq, Ws, N, K)
    wb = synth.weights_bf16(256, K, synth.CFG_SKINNY).to(dev)
    gu = synth.activations(M, 2 * K, synth.CFG_TINY).to(dev)
    # outputs and workspaces allocated before capture
    q = torch.empty((M, K), dtype=torch.uint8, device=dev)
    s = torch.empty((M,), dtype=torch.float32, device=dev)
    qg = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sg = torch.empty((M, K // 128), dtype=torch.float32, device=dev)
    c1 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    c2 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    c3 = torch.empty((M, 256), dtype=torch.bfloat16, device=dev)
    q2 = torch.empty((M, K), dtype=torch.uint8, device=dev)
    s2 = torch.empty((M,), dtype=torch.float32, device=dev)
    ro = torch.empty_like(res)
    q3 = torch.empty((M, K), dtype=torch.uint8, device=dev)
    s3 = torch.empty((M,), dtype=torch.float32, device=dev)
    ws1 = r4q.workspace(r4q.R4_OP_W4A8_MXFP4, M, N, K, dev)
    ws3 = r4q.workspace(r4q.R4_OP_LINEAR_W4A8_MXFP4, M, N, K, dev)
    c5 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    c6 = torch.zeros((M, N), dtype=torch.bfloat16, device=dev)   # row M-1 is never written
    ws2 = r4q.workspace(r4q.R4_OP_BLOCKFP8, M, N, K, dev)
    c4 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

    def step():
        r4q.r4_quant_fp8_per_token(x, M, K, K, K, q, s)
        r4q.r4_quant_fp8_per_token(x, M, K, K, 128, qg, sg)
        r4q.r4_gemm_w4a8_mxfp4(q, s, pk, M, N, K, c1, N, ws1)
        r4q.r4_linear_w4a8_mxfp4(x, K, pk, M, N, K, c5, N, ws3)             # quantizer + GEMM
        r4q.r4_linear_w4a8_mxfp4(x[:M - 1], K, pk, M - 1, N, K, c6, N, ws3)  # 15 tokens, same workspace
        r4q.r4_gemm_blockfp8(qg, sg, pk8, M, N, K, c2, N, ws2)
        r4q.r4_gemm_bf16_nt_skinny(x, wb, M, 256, K, c3, 256)
        r4q.r4_add_rmsnorm_quant_fp8(x, res, nw, 1e-6, M, K, ro, q2, s2)
        r4q.r4_silu_mul_quant_fp8(gu, M, K, q3, s3)
        # the no-allocation GEMM on a split-K schedule, so that its clearing
        # of the static scratch and the split-K reduction are in the graph
        # (the eager call below also looks up the scratch address first)
        r4q.r4_set_option(1, 4)
        r4q.r4_set_option(6, 0)
        try:
            r4q.r4_gemm_w4a8_mxfp4_noalloc(q, s, pk, M, N, K, c4, N)
        finally:
            r4q.r4_set_option(1, 0)
            r4q.r4_set_option(6, 1)

    outs = (q, s, qg, sg, c1, c2, c3, q2, s2, ro, q3, s3, c4, c5, c6)
    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in outs]
    for t in outs:
        t.zero_()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            step()
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    assert r4q.r4_device_error(clear=True) == 0
    for a, b in zip(eager, outs):
        assert torch.equal(a, b)
