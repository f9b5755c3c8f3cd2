"""Seeded synthetic inputs for the quantized linear path.

This module only draws random numbers: it holds none of the method's
arithmetic (no quantization, no scaling, no encoding), so the CUDA path and
the CPU oracle can both be fed from it without sharing any of the computation
under test. Everything is generated on the CPU with ``torch.Generator`` so the
same seed gives the same tensor on any machine.

Workloads and value distributions
---------------------------------
* activations: x ~ N(0, 1), cast to bfloat16. With ``outliers=True``,
  ceil(0.01 K) channels, picked by ``randperm(K)`` from their own seed, are
  multiplied by 20 on every row before the cast (outlier channels, the usual
  shape of LLM activations entering a quantized linear layer).
* weights: W ~ N(0, 0.02) in float32, the master copy that a checkpoint
  quantizer would turn into MXFP4 or block-FP8.
* skinny weights: W ~ N(0, 0.02) cast to bfloat16.

Seeds: activations 1000 + cfg, weights 2000 + cfg, outlier channels 3000 + cfg,
where cfg is the workload number (1 tiny W4A8, 2 decode W4A8, 3 prefill W4A8,
4 block-FP8, 5 skinny bf16). Activations are drawn row-major, so the first M
rows of a tall draw equal a short draw of M rows with the same seed.
"""

import math

import torch

CFG_TINY, CFG_DECODE, CFG_PREFILL, CFG_BLOCKFP8, CFG_SKINNY = 1, 2, 3, 4, 5

# Shapes of each workload: (N, K) pairs and the token counts M.
TINY = dict(M=8, N=256, K=2048)
DECODE_M = (6, 8, 16, 32, 64)
DECODE_NK = ((34816, 5120), (5120, 17408), (2048, 5120))
PREFILL_M = (256, 2048, 8192)
PREFILL_NK = ((34816, 5120), (5120, 17408), (10240, 5120))
BLOCKFP8_M = (8, 64, 2048)
BLOCKFP8_NK = ((6144, 2048), (2048, 6144), (4096, 4096))
SKINNY_M = (6, 8, 16, 32, 64)
SKINNY_NK = ((256, 2048), (96, 5120))


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def outlier_channels(K, cfg):
    """Indices of the ceil(0.01 K) outlier channels for workload ``cfg``."""
    n = math.ceil(0.01 * K)
    return torch.randperm(K, generator=_gen(3000 + cfg))[:n]


def activations(M, K, cfg, outliers=False, seed=None):
    """x [M, K] bfloat16 (CPU), N(0,1) with optional x20 outlier channels."""
    g = _gen(1000 + cfg if seed is None else seed)
    x = torch.randn(M, K, generator=g, dtype=torch.float32)
    if outliers:
        x[:, outlier_channels(K, cfg)] *= 20.0
    return x.to(torch.bfloat16)


def weights_fp32(N, K, cfg, std=0.02, seed=None):
    """W [N, K] float32 (CPU) ~ N(0, std)."""
    g = _gen(2000 + cfg if seed is None else seed)
    return torch.randn(N, K, generator=g, dtype=torch.float32) * std


def weights_bf16(N, K, cfg, std=0.02, seed=None):
    """W [N, K] bfloat16 (CPU) ~ N(0, std), for the skinny GEMM."""
    return weights_fp32(N, K, cfg, std=std, seed=seed).to(torch.bfloat16)


def uniform_bytes(shape, seed, low=0, high=256):
    """Uniform random integers in [low, high) as uint8 (CPU)."""
    g = _gen(seed)
    return torch.randint(low, high, shape, generator=g, dtype=torch.int64).to(torch.uint8)


def sample_indices(n, count, seed):
    """``count`` distinct sorted indices in [0, n) (for sampled parity checks)."""
    count = min(n, count)
    return torch.randperm(n, generator=_gen(seed))[:count].sort().values
