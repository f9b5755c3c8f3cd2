"""CPU oracle for the block-scaled quantized linear path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library and its
Python binding) may import, call or link anything in this package. Only the test
suite, the smoke check and the CPU-baseline leg of the benchmark use it.

What it is: a plain, slow, obviously correct restatement of what the pages
compute, in NumPy, with every product and sum formed in float64 and one final
rounding to bfloat16. It shares no code, table or constant with the CUDA path.

Sources (page title, then the section on it):
  * radiance_mxfp4.py -- module docstring (W4A8: e2m1 weights + ue8m0 scale per
    32 K, per-token e4m3 activations), ``_traced_quant`` and the comment above it
    (per-token quantization rule), ``_exact_ref`` (e2m1 value table, nibble order,
    2^(s-127) scale decode, dequantize-then-multiply reference).
  * radiance_kernels.py -- ``block_scaled_mm`` and the preshuffle load hook
    (block-FP8 W8A8: e4m3 weights with one fp32 scale per 128x128 block,
    activations with one scale per token per 128 K).
  * radiance_gemm.py -- module docstring (skinny bf16 NT GEMM C = x W^T with
    fp32 accumulation).
  * radiance_arnq.py -- module docstring, ``ar_add_rms_quant``,
    ``silu_mul_quant`` and the ``_SiluMulQuant`` docstring (fused residual-add
    + RMS norm + quant and SiluAndMul + quant producers).

Modules:
  formats -- value tables and round-to-nearest-even encoders for e4m3, e2m1,
             ue8m0 and bfloat16.
  quant   -- activation quantization (per token, per 128-K group) and the
             weight quantizers used only to manufacture test inputs.
  gemm    -- the three GEMM definitions.
  fused   -- the fused quantization producers (add + RMS norm + quant,
             SiluAndMul + quant).
"""

from . import formats, quant, gemm, fused  # noqa: F401
