"""The GEMM planners' schedules through r4_plan_gemm (host arithmetic, no GPU).

The block-FP8 planner touches no device, so its rules are checked exactly;
for W4A8/W4A4 the checks hold whether or not a device answers the cluster
query (without one, no cluster split is taken)."""

import itertools

import pytest

from block_scaled_precision_token_gb300 import r4q

FP8, W4A8, W4A4, LINEAR = r4q.R4_OP_BLOCKFP8, r4q.R4_OP_W4A8_MXFP4, r4q.R4_OP_W4A4_MXFP4, r4q.R4_OP_LINEAR_W4A8_MXFP4


@pytest.fixture(autouse=True)
def _options_reset():
    yield
    for key, default in ((1, 0), (3, 0), (7, 0), (8, 0)):
        r4q.r4_set_option(key, default)


def plan(op, M, N, K, sms=152):
    return r4q.r4_plan_gemm(op, M, N, K, sms)


def _consistent(p, M, N, K):
    """What every schedule must satisfy: the tiles cover C, the K splits
    cover K with no empty split, and the grid has work for every CTA."""
    KB = -(-K // 128)
    assert p["token_tile"] * p["t_tiles"] >= M > p["token_tile"] * (p["t_tiles"] - 1)
    assert p["weight_rows"] * p["n_tiles"] >= N > p["weight_rows"] * (p["n_tiles"] - 1)
    if not p["stream_k"]:
        assert p["splits"] * p["kb_per_split"] >= KB > (p["splits"] - 1) * p["kb_per_split"]
        assert p["units"] == p["n_tiles"] * p["t_tiles"] * p["splits"]
        assert 1 <= p["grid"] <= p["units"]


def test_blockfp8_weight_rows():
    """256 weight rows for the 128-token tile when N allows and the 256-row
    tiles fill at least half of the SMs; else 128."""
    p = plan(FP8, 2048, 6144, 2048)
    assert (p["token_tile"], p["weight_rows"], p["n_tiles"], p["t_tiles"]) == (128, 256, 24, 16)
    assert (p["splits"], p["units"], p["grid"]) == (1, 384, 152)
    assert plan(FP8, 512, 6144, 2048)["weight_rows"] == 256        # 24 x 4 = 96 tiles >= 76
    assert plan(FP8, 256, 6144, 2048)["weight_rows"] == 128        # 24 x 2 = 48 < 76
    assert plan(FP8, 2048, 6016, 2048)["weight_rows"] == 128       # N not a multiple of 256
    assert plan(FP8, 64, 6144, 2048)["weight_rows"] == 128         # decode tiles keep weights on the lanes
    r4q.r4_set_option(8, 128)
    assert plan(FP8, 2048, 6144, 2048)["weight_rows"] == 128
    r4q.r4_set_option(8, 256)
    assert plan(FP8, 256, 6144, 2048)["weight_rows"] == 256
    assert plan(FP8, 2048, 6016, 2048)["weight_rows"] == 128       # forcing cannot break the tiling


def test_blockfp8_token_tiles_and_decode_splits():
    """16 tokens up to 16, two 32-token tiles for 33-64, 128 above; decode
    tiles split K as far as keeps every unit in one wave."""
    assert plan(FP8, 16, 2048, 6144)["token_tile"] == 16
    p = plan(FP8, 64, 4096, 4096)
    assert (p["token_tile"], p["t_tiles"]) == (32, 2)
    assert plan(FP8, 65, 4096, 4096)["token_tile"] == 128
    p = plan(FP8, 8, 6144, 2048)
    assert (p["n_tiles"], p["splits"], p["kb_per_split"], p["units"], p["grid"]) == (48, 3, 6, 144, 144)
    for sms in (132, 148, 152):
        for N, K in ((6144, 2048), (2048, 6144), (4096, 4096)):
            p = plan(FP8, 8, N, K, sms)
            assert p["units"] <= sms


def test_blockfp8_prefill_splits():
    """128-token tiles stay unsplit while they fill a quarter of the SMs; a
    forced factor is rounded to a schedule without an empty split; more
    tiles than the counter region holds never split."""
    assert plan(FP8, 2048, 2048, 6144)["splits"] == 1
    assert plan(FP8, 256, 6144, 2048)["splits"] == 1                 # 48 x 2 = 96 tiles >= 38
    p = plan(FP8, 256, 2048, 6144)                                   # 16 x 2 = 32 tiles < 38: the wave model
    assert p["splits"] > 1 and p["units"] <= 152                     # splits, within one wave
    r4q.r4_set_option(3, 5)
    p = plan(FP8, 200, 384, 2048)
    assert p["splits"] == 4 and p["kb_per_split"] == 4               # 16 K blocks: 5 would leave 4,4,4,4,0
    r4q.r4_set_option(3, 2)
    assert plan(FP8, 8, 128 * 4097, 256)["splits"] == 1              # 4097 tiles > the 4096 counters


def test_w4a8_prefill_forced_split_clamped():
    """Prefill tiles split only with at most one split unit per CTA, forced
    factors included (272 tiles x 16 splits would put several on each)."""
    r4q.r4_set_option(1, 16)
    for op in (W4A8, W4A4, LINEAR):
        p = plan(op, 256, 34816, 5120)
        assert p["token_tile"] >= 128 and p["splits"] == 1


@pytest.mark.parametrize("op", [FP8, W4A8, W4A4])
def test_schedules_consistent(op):
    Ms = (1, 6, 16, 33, 64, 65, 200, 256, 2048, 8192)
    NKs = ((2048, 5120), (5120, 17408), (34816, 5120), (6144, 2048), (384, 1024))
    for (M, (N, K)), sms in itertools.product(itertools.product(Ms, NKs), (132, 152)):
        _consistent(plan(op, M, N, K, sms), M, N, K)


def test_plan_arguments():
    lib = r4q.lib()
    out = (r4q.ctypes.c_int32 * 10)()
    ptr = r4q.ctypes.cast(out, r4q.ctypes.c_void_p)
    assert lib.r4_plan_gemm(FP8, 8, 6144, 2048, 152, None) == r4q.R4_ERR_INVALID_ARG
    assert lib.r4_plan_gemm(FP8, 0, 6144, 2048, 152, ptr) == r4q.R4_ERR_INVALID_ARG
    assert lib.r4_plan_gemm(FP8, 8, 6144, 2048, 0, ptr) == r4q.R4_ERR_INVALID_ARG
    assert lib.r4_plan_gemm(r4q.R4_OP_BF16_SKINNY, 8, 256, 2048, 152, ptr) == r4q.R4_ERR_INVALID_ARG
    assert lib.r4_plan_gemm(FP8, 8, 6100, 2048, 152, ptr) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert lib.r4_plan_gemm(W4A8, 8, 6144, 96, 152, ptr) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert lib.r4_plan_gemm(FP8, 8, 6144, 2048, 152, ptr) == 0 and out[0] == 16
