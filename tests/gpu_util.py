"""Helpers for the GPU parity tests (test infrastructure)."""

import numpy as np
import pytest
import torch

from oracle import gemm as G


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from block_scaled_precision_token_gb300 import build
    build.build()
    from block_scaled_precision_token_gb300 import r4q
    r4q.lib()
    return r4q


def np_u8(t):
    return t.detach().cpu().numpy().astype(np.uint8)


def np_f32(t):
    return t.detach().float().cpu().numpy()


def bf16_to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_gemm_matches(out_bf16, c64, what=""):
    """Elementwise: |gpu - exact| <= 4e-3 |exact| + 1e-3 rms(exact row), and the
    page's relative Frobenius error well below its 0.02 'wrong' line."""
    got = bf16_to_np(out_bf16)
    assert got.shape == c64.shape, (got.shape, c64.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    ok, ratio = G.gemm_tolerance_ok(got, c64)
    rel = G.rel_frobenius(got, c64)
    assert ok, f"{what}: worst error/bound = {ratio:.3f}, rel_frobenius = {rel:.3e}"
    assert rel < 5e-3, f"{what}: rel_frobenius = {rel:.3e}"
    return ratio, rel


def check_device_error(r4q):
    torch.cuda.synchronize()
    code = r4q.r4_device_error(clear=True)
    assert code == 0, f"a kernel reported a timed-out device wait (code {code})"


def random_e4m3_codes(shape, seed):
    """Uniform finite e4m3 codes (NaN codes 0x7F / 0xFF replaced)."""
    from block_scaled_precision_token_gb300 import synth
    q = synth.uniform_bytes(shape, seed).numpy()
    q[(q & 0x7F) == 0x7F] = 0x3C
    return q


def prepack_inverse_mxfp4(packed, N, K):
    """Test-only inverse of the MXFP4 prepack: returns (codes [N, K/2], scales
    [N, K/32], padding_ok)."""
    NT, KB = -(-N // 128), -(-K // 128)
    p = np.asarray(packed, dtype=np.uint8)
    nc = NT * KB * 8192
    codes = p[:nc].reshape(NT, KB, 128, 64).transpose(0, 2, 1, 3).reshape(NT * 128, KB * 64)
    sf = p[nc:nc + NT * KB * 512].reshape(NT, KB, 32, 4, 4)       # [nt][kb][r0][r1][j]
    sf = sf.transpose(0, 3, 2, 1, 4).reshape(NT * 128, KB * 4)     # row = 32 r1 + r0
    pad_ok = (np.all(codes[N:] == 0) and np.all(codes[:, K // 2:] == 0)
              and np.all(sf[N:] == 127) and np.all(sf[:, K // 32:] == 127))
    return codes[:N, :K // 2], sf[:N, :K // 32], pad_ok


def prepack_inverse_blockfp8(packed, N, K):
    NT, KB = N // 128, K // 128
    p = np.asarray(packed, dtype=np.uint8)
    codes = p[:N * K].reshape(NT, KB, 128, 128).transpose(0, 2, 1, 3).reshape(N, K)
    sc = p[N * K:N * K + NT * KB * 4].view(np.float32).reshape(NT, KB)
    return codes, sc
