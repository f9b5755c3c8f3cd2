"""The C-ABI library builds, loads, exports every entry point the header
declares, and rejects bad arguments on the host (no GPU needed)."""

import ctypes
import math

import pytest

from block_scaled_precision_token_gb300 import build as B


@pytest.fixture(scope="module")
def r4q():
    B.build()
    from block_scaled_precision_token_gb300 import r4q as mod
    mod.lib()
    return mod


def test_every_header_symbol_is_exported(r4q):
    syms = r4q.header_symbols()
    assert len(syms) >= 16
    lib = r4q.lib()
    for name in syms:
        assert hasattr(lib, name), name
    assert set(syms) == set(r4q._SIGS), "binding and header disagree"


def test_version_and_strings(r4q):
    assert r4q.r4_version() >= 1
    for st in range(7):
        assert r4q.status_string(st) and r4q.status_string(st) != "unknown status"
    assert r4q.status_string(99) == "unknown status"


def test_prepack_sizes(r4q):
    lib = r4q.lib()
    for N, K in [(256, 2048), (34816, 5120), (300, 416), (1, 32)]:
        want = math.ceil(N / 128) * math.ceil(K / 128) * (8192 + 512)
        assert lib.r4_prepack_mxfp4_bytes(N, K) == want
    assert lib.r4_prepack_mxfp4_bytes(256, 48) == 0          # K % 32
    assert lib.r4_prepack_blockfp8_bytes(6144, 2048) == 6144 * 2048 + 48 * 16 * 4
    assert lib.r4_prepack_blockfp8_bytes(100, 2048) == 0


def test_options(r4q):
    lib = r4q.lib()
    assert lib.r4_set_option(99, 0) == r4q.R4_ERR_INVALID_ARG
    assert lib.r4_set_option(9, 1) == r4q.R4_ERR_INVALID_ARG   # unassigned
    assert lib.r4_set_option(2, 48) == r4q.R4_ERR_INVALID_ARG
    assert lib.r4_set_option(2, 64) == 0 and lib.r4_set_option(2, 0) == 0
    assert lib.r4_set_option(2, 192) == 0 and lib.r4_set_option(2, 0) == 0
    assert lib.r4_set_option(2, 160) == r4q.R4_ERR_INVALID_ARG
    assert lib.r4_set_option(16, 3) == r4q.R4_ERR_INVALID_ARG and lib.r4_set_option(16, -1) == r4q.R4_ERR_INVALID_ARG
    assert lib.r4_set_option(16, 2) == 0 and lib.r4_set_option(16, 1) == 0 and lib.r4_set_option(16, 0) == 0
    assert lib.r4_set_option(1, 0) == 0 and lib.r4_set_option(3, 0) == 0


def test_validation_rejects_before_launch(r4q):
    lib = r4q.lib()
    P = ctypes.c_void_p
    good = P(1 << 20)           # never dereferenced: validation fails first
    odd = P((1 << 20) + 8)      # 8-byte aligned, not 16
    S = P(0)
    # null pointers
    assert lib.r4_quant_fp8_per_token(None, 8, 2048, 2048, 2048, good, good, S) == r4q.R4_ERR_INVALID_ARG
    assert lib.r4_gemm_w4a8_mxfp4(good, good, None, 8, 256, 2048, good, 256, None, 0, S) == r4q.R4_ERR_INVALID_ARG
    assert lib.r4_gemm_bf16_nt_skinny(None, good, 8, 256, 2048, good, 256, None, 0, S) == r4q.R4_ERR_INVALID_ARG
    # bad sizes
    assert lib.r4_quant_fp8_per_token(good, 0, 2048, 2048, 2048, good, good, S) == r4q.R4_ERR_INVALID_ARG
    assert lib.r4_quant_fp8_per_token(good, 8, 2048, 1024, 2048, good, good, S) == r4q.R4_ERR_INVALID_ARG
    assert lib.r4_gemm_w4a8_mxfp4(good, good, good, 8, 256, 2048, good, 100, None, 0, S) == r4q.R4_ERR_INVALID_ARG
    # unsupported shapes
    assert lib.r4_quant_fp8_per_token(good, 8, 2044, 2048, 2044, good, good, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert lib.r4_quant_fp8_per_token(good, 8, 2048, 2048, 64, good, good, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert lib.r4_gemm_w4a8_mxfp4(good, good, good, 8, 256, 2000, good, 256, None, 0, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert lib.r4_gemm_blockfp8(good, good, good, 8, 200, 2048, good, 200, None, 0, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert lib.r4_gemm_bf16_nt_skinny(good, good, 65, 256, 2048, good, 256, None, 0, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert lib.r4_gemm_bf16_nt_skinny(good, good, 8, 256, 2000, good, 256, None, 0, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert lib.r4_prepack_blockfp8(good, good, 200, 256, good, 1 << 30, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    # misalignment
    assert lib.r4_quant_fp8_per_token(odd, 8, 2048, 2048, 2048, good, good, S) == r4q.R4_ERR_MISALIGNED
    assert lib.r4_prepack_mxfp4(good, good, 256, 2048, odd, 1 << 30, S) == r4q.R4_ERR_MISALIGNED
    assert lib.r4_gemm_w4a8_mxfp4(good, good, odd, 8, 256, 2048, good, 256, None, 0, S) == r4q.R4_ERR_MISALIGNED
    # short prepack buffer
    assert lib.r4_prepack_mxfp4(good, good, 256, 2048, good, 100, S) == r4q.R4_ERR_WORKSPACE
    assert lib.r4_prepack_blockfp8(good, good, 256, 256, good, 100, S) == r4q.R4_ERR_WORKSPACE


def test_validation_of_the_later_entry_points(r4q):
    """Fused producers, the no-allocation GEMM and the quotient self-check
    reject bad arguments on the host, before any device work."""
    lib = r4q.lib()
    P = ctypes.c_void_p
    good = P(1 << 20)
    odd8 = P((1 << 20) + 8)
    odd4 = P((1 << 20) + 4)
    S = P(0)
    f = ctypes.c_float
    arq = lib.r4_add_rmsnorm_quant_fp8
    assert arq(None, good, good, f(1e-6), 8, 5120, good, good, good, S) == r4q.R4_ERR_INVALID_ARG
    assert arq(good, good, good, f(1e-6), 0, 5120, good, good, good, S) == r4q.R4_ERR_INVALID_ARG
    assert arq(good, good, good, f(-1.0), 8, 5120, good, good, good, S) == r4q.R4_ERR_INVALID_ARG
    assert arq(good, good, good, f(float("nan")), 8, 5120, good, good, good, S) == r4q.R4_ERR_INVALID_ARG
    assert arq(good, good, good, f(1e-6), 8, 5124, good, good, good, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert arq(good, good, good, f(1e-6), 8, 24584, good, good, good, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert arq(odd8, good, good, f(1e-6), 8, 5120, good, good, good, S) == r4q.R4_ERR_MISALIGNED
    assert arq(good, good, good, f(1e-6), 8, 5120, good, odd4, good, S) == r4q.R4_ERR_MISALIGNED
    smq = lib.r4_silu_mul_quant_fp8
    assert smq(None, 8, 17408, good, good, S) == r4q.R4_ERR_INVALID_ARG
    assert smq(good, 0, 17408, good, good, S) == r4q.R4_ERR_INVALID_ARG
    assert smq(good, 8, 17412, good, good, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert smq(good, 8, 24584, good, good, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert smq(odd8, 8, 17408, good, good, S) == r4q.R4_ERR_MISALIGNED
    na = lib.r4_gemm_w4a8_mxfp4_noalloc
    assert na(good, good, None, 8, 256, 2048, good, 256, S) == r4q.R4_ERR_INVALID_ARG
    assert na(good, good, good, 8, 256, 2048, good, 100, S) == r4q.R4_ERR_INVALID_ARG
    assert na(good, good, good, 8, 256, 2000, good, 256, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert na(good, good, odd8, 8, 256, 2048, good, 256, S) == r4q.R4_ERR_MISALIGNED
    assert na(odd8, good, good, 8, 256, 2048, good, 256, S) == r4q.R4_ERR_MISALIGNED
    ln = lib.r4_linear_w4a8_mxfp4
    assert ln(None, 2048, good, 8, 256, 2048, good, 256, good, 1 << 20, S) == r4q.R4_ERR_INVALID_ARG
    assert ln(good, 2048, good, 8, 256, 2048, good, 100, good, 1 << 20, S) == r4q.R4_ERR_INVALID_ARG
    assert ln(good, 1024, good, 8, 256, 2048, good, 256, good, 1 << 20, S) == r4q.R4_ERR_INVALID_ARG
    assert ln(good, 0, good, 0, 256, 2048, good, 256, good, 1 << 20, S) == r4q.R4_ERR_INVALID_ARG
    assert ln(good, 2000, good, 8, 256, 2000, good, 256, good, 1 << 20, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert ln(good, 2052, good, 8, 256, 2048, good, 256, good, 1 << 20, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert ln(good, 2048, odd8, 8, 256, 2048, good, 256, good, 1 << 20, S) == r4q.R4_ERR_MISALIGNED
    assert lib.r4_check_quotients(None, good, S) == r4q.R4_ERR_INVALID_ARG
    assert lib.r4_check_quotients(odd4, good, S) == r4q.R4_ERR_MISALIGNED


def test_validation_of_the_w4a4_entry_points_and_the_probe(r4q):
    """The MXFP4 activation quantizer, the W4A4 GEMM and the MMA issue-rate
    probe reject bad arguments on the host, before any device work; the
    scale-buffer size query follows the documented atom layout."""
    lib = r4q.lib()
    P = ctypes.c_void_p
    good = P(1 << 20)
    odd8 = P((1 << 20) + 8)
    S = P(0)
    # scale atoms: tokens padded to 256, K to 128, 512 bytes per 128 x 128
    for M, K in [(8, 5120), (256, 2048), (257, 416), (2048, 17408)]:
        want = math.ceil(M / 256) * 2 * math.ceil(K / 128) * 512
        assert lib.r4_quant_mxfp4_act_scale_bytes(M, K) == want
    assert lib.r4_quant_mxfp4_act_scale_bytes(8, 48) == 0
    assert lib.r4_quant_mxfp4_act_scale_bytes(0, 128) == 0
    qa = lib.r4_quant_mxfp4_act
    big = 1 << 30
    assert qa(None, 8, 2048, 2048, good, good, big, S) == r4q.R4_ERR_INVALID_ARG
    assert qa(good, 0, 2048, 2048, good, good, big, S) == r4q.R4_ERR_INVALID_ARG
    assert qa(good, 8, 2048, 1024, good, good, big, S) == r4q.R4_ERR_INVALID_ARG
    assert qa(good, 8, 2000, 2000, good, good, big, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert qa(good, 8, 2048, 2052, good, good, big, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert qa(odd8, 8, 2048, 2048, good, good, big, S) == r4q.R4_ERR_MISALIGNED
    assert qa(good, 8, 2048, 2048, good, odd8, big, S) == r4q.R4_ERR_MISALIGNED
    assert qa(good, 8, 2048, 2048, good, good, 100, S) == r4q.R4_ERR_WORKSPACE
    g4 = lib.r4_gemm_w4a4_mxfp4
    assert g4(good, None, good, 8, 256, 2048, good, 256, None, 0, S) == r4q.R4_ERR_INVALID_ARG
    assert g4(good, good, good, 8, 256, 2048, good, 100, None, 0, S) == r4q.R4_ERR_INVALID_ARG
    assert g4(good, good, good, 8, 256, 2000, good, 256, None, 0, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert g4(good, good, good, 8, 256, 96, good, 256, None, 0, S) == r4q.R4_ERR_UNSUPPORTED_SHAPE
    assert g4(good, odd8, good, 8, 256, 2048, good, 256, None, 0, S) == r4q.R4_ERR_MISALIGNED
    assert g4(good, good, odd8, 8, 256, 2048, good, 256, None, 0, S) == r4q.R4_ERR_MISALIGNED
    pk = lib.r4_mma_peak
    for kind, n, blocks, iters in [(0, 256, 152, 10), (4, 256, 152, 10), (1, 192, 152, 10), (1, 256, 0, 10),
                                   (1, 256, 70000, 10), (1, 256, 152, 0)]:
        assert pk(kind, n, blocks, iters, S) == r4q.R4_ERR_INVALID_ARG, (kind, n, blocks, iters)


def test_row_kernel_options(r4q):
    lib = r4q.lib()
    for key, bad, ok in [(11, 3, 8), (11, 16, 1), (13, 96, 128), (13, 512, 64), (5, 3, 1), (5, -1, 2),
                         (15, 5, 1), (15, -1, 4), (8, 64, 256), (8, 192, 128)]:
        assert lib.r4_set_option(key, bad) == r4q.R4_ERR_INVALID_ARG
        assert lib.r4_set_option(key, ok) == 0
        assert lib.r4_set_option(key, 0) == 0
    assert lib.r4_set_option(5, 2) == 0          # the default: rolling L2 prefetch
    assert lib.r4_set_option(14, 0) == 0 and lib.r4_set_option(14, 1) == 0


def test_product_path_has_no_oracle_import():
    """The package must not import the oracle (or any CPU fallback)."""
    import ast
    import os
    pkg = os.path.dirname(B.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith(".py"):
                tree = ast.parse(open(os.path.join(root, f)).read())
                for node in ast.walk(tree):
                    if isinstance(node, ast.Import):
                        assert not any(a.name.split(".")[0] == "oracle" for a in node.names), f
                    if isinstance(node, ast.ImportFrom):
                        assert (node.module or "").split(".")[0] != "oracle", f
