"""Thin ctypes binding of libr4q.so (the C ABI in include/r4q.h).

Each ``r4_*`` function here has the name of the C entry point it wraps and
does argument marshalling only: it takes torch tensors for the pointer
arguments (device memory owned by the caller), passes ``data_ptr()`` and the
sizes through, launches on the current torch CUDA stream, and raises
``R4Error`` on a non-zero status. All arithmetic runs in the library's CUDA
kernels; there is no fallback path. The convenience helpers at the end
(``quant_fp8``, ``prepack_mxfp4``, ``gemm_w4a8`` ...) only allocate outputs with
torch and call the bindings.
"""

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libr4q.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "r4q.h")

R4_OK, R4_ERR_INVALID_ARG, R4_ERR_UNSUPPORTED_SHAPE, R4_ERR_MISALIGNED = 0, 1, 2, 3
R4_ERR_WORKSPACE, R4_ERR_CUDA, R4_ERR_DEVICE_TIMEOUT = 4, 5, 6
R4_OP_W4A8_MXFP4, R4_OP_BLOCKFP8, R4_OP_BF16_SKINNY, R4_OP_W4A4_MXFP4, R4_OP_LINEAR_W4A8_MXFP4 = 1, 2, 3, 4, 5


class R4Error(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


_lib = None
_P, _I64, _I, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t

_SIGS = {
    "r4_version": ([], _I),
    "r4_status_string": ([_I], ctypes.c_char_p),
    "r4_last_kernel_name": ([], ctypes.c_char_p),
    "r4_device_error": ([_P, _I], _I),
    "r4_set_option": ([_I, _I64], _I),
    "r4_quant_fp8_per_token": ([_P, _I64, _I64, _I64, _I64, _P, _P, _P], _I),
    "r4_quantize_mxfp4_weight": ([_P, _I64, _I64, _P, _P, _P], _I),
    "r4_quantize_blockfp8_weight": ([_P, _I64, _I64, _P, _P, _P], _I),
    "r4_prepack_mxfp4_bytes": ([_I64, _I64], _SZ),
    "r4_prepack_mxfp4": ([_P, _P, _I64, _I64, _P, _SZ, _P], _I),
    "r4_prepack_blockfp8_bytes": ([_I64, _I64], _SZ),
    "r4_prepack_blockfp8": ([_P, _P, _I64, _I64, _P, _SZ, _P], _I),
    "r4_gemm_workspace_bytes": ([_I, _I64, _I64, _I64], _SZ),
    "r4_plan_gemm": ([_I, _I64, _I64, _I64, _I, _P], _I),
    "r4_gemm_w4a8_mxfp4": ([_P, _P, _P, _I64, _I64, _I64, _P, _I64, _P, _SZ, _P], _I),
    "r4_linear_w4a8_mxfp4": ([_P, _I64, _P, _I64, _I64, _I64, _P, _I64, _P, _SZ, _P], _I),
    "r4_gemm_blockfp8": ([_P, _P, _P, _I64, _I64, _I64, _P, _I64, _P, _SZ, _P], _I),
    "r4_gemm_bf16_nt_skinny": ([_P, _P, _I64, _I64, _I64, _P, _I64, _P, _SZ, _P], _I),
    "r4_gemm_w4a8_mxfp4_noalloc": ([_P, _P, _P, _I64, _I64, _I64, _P, _I64, _P], _I),
    "r4_add_rmsnorm_quant_fp8": ([_P, _P, _P, ctypes.c_float, _I64, _I64, _P, _P, _P, _P], _I),
    "r4_silu_mul_quant_fp8": ([_P, _I64, _I64, _P, _P, _P], _I),
    "r4_check_quotients": ([_P, _P, _P], _I),
    "r4_mma_peak": ([_I, _I, _I, _I, _P], _I),
    "r4_quant_mxfp4_act_scale_bytes": ([_I64, _I64], _SZ),
    "r4_quant_mxfp4_act": ([_P, _I64, _I64, _I64, _P, _P, _SZ, _P], _I),
    "r4_gemm_w4a4_mxfp4": ([_P, _P, _P, _I64, _I64, _I64, _P, _I64, _P, _SZ, _P], _I),
}


def lib():
    """Load libr4q.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m block_scaled_precision_token_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _lib = handle
    return _lib


def header_symbols():
    """Entry points declared in include/r4q.h."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char|void)\s*\*?\s*(r4_\w+)\s*\(",
                                 text, flags=re.M)))


def status_string(status):
    return lib().r4_status_string(int(status)).decode()


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _check(status, where):
    if status != R4_OK:
        raise R4Error(status, where)


def _need(t, dtype, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


# --------------------------------------------------------------------------- bindings

def r4_version():
    return lib().r4_version()


def r4_last_kernel_name():
    return lib().r4_last_kernel_name().decode()


def r4_set_option(key, value):
    _check(lib().r4_set_option(int(key), int(value)), "r4_set_option")


def r4_device_error(clear=True):
    """Device error word of the current device (0 = no kernel reported a timeout)."""
    v = ctypes.c_int(0)
    st = lib().r4_device_error(ctypes.byref(v), 1 if clear else 0)
    if st not in (R4_OK, R4_ERR_DEVICE_TIMEOUT):
        raise R4Error(st, "r4_device_error")
    return v.value


def r4_quant_fp8_per_token(x, M, K, ldx, group, q, s, stream=None):
    _need(x, torch.bfloat16, "x"); _need(q, torch.uint8, "q"); _need(s, torch.float32, "s")
    _check(lib().r4_quant_fp8_per_token(_ptr(x), M, K, ldx, group, _ptr(q), _ptr(s), _stream(stream)),
           "r4_quant_fp8_per_token")


def r4_quantize_mxfp4_weight(w, N, K, packed, scale, stream=None):
    _need(w, torch.float32, "w"); _need(packed, torch.uint8, "packed"); _need(scale, torch.uint8, "scale")
    _check(lib().r4_quantize_mxfp4_weight(_ptr(w), N, K, _ptr(packed), _ptr(scale), _stream(stream)),
           "r4_quantize_mxfp4_weight")


def r4_quantize_blockfp8_weight(w, N, K, q, s, stream=None):
    _need(w, torch.float32, "w"); _need(q, torch.uint8, "q"); _need(s, torch.float32, "s")
    _check(lib().r4_quantize_blockfp8_weight(_ptr(w), N, K, _ptr(q), _ptr(s), _stream(stream)),
           "r4_quantize_blockfp8_weight")


def r4_quant_mxfp4_act_scale_bytes(M, K):
    return int(lib().r4_quant_mxfp4_act_scale_bytes(M, K))


def r4_quant_mxfp4_act(x, M, K, ldx, q, scale, stream=None):
    _need(x, torch.bfloat16, "x"); _need(q, torch.uint8, "q"); _need(scale, torch.uint8, "scale")
    _check(lib().r4_quant_mxfp4_act(_ptr(x), M, K, ldx, _ptr(q), _ptr(scale), scale.numel(), _stream(stream)),
           "r4_quant_mxfp4_act")


def r4_prepack_mxfp4_bytes(N, K):
    return int(lib().r4_prepack_mxfp4_bytes(N, K))


def r4_prepack_mxfp4(w, w_scale, N, K, packed, stream=None):
    _need(w, torch.uint8, "w"); _need(w_scale, torch.uint8, "w_scale"); _need(packed, torch.uint8, "packed")
    _check(lib().r4_prepack_mxfp4(_ptr(w), _ptr(w_scale), N, K, _ptr(packed), packed.numel(), _stream(stream)),
           "r4_prepack_mxfp4")


def r4_prepack_blockfp8_bytes(N, K):
    return int(lib().r4_prepack_blockfp8_bytes(N, K))


def r4_prepack_blockfp8(w, w_scale, N, K, packed, stream=None):
    _need(w, torch.uint8, "w"); _need(w_scale, torch.float32, "w_scale"); _need(packed, torch.uint8, "packed")
    _check(lib().r4_prepack_blockfp8(_ptr(w), _ptr(w_scale), N, K, _ptr(packed), packed.numel(), _stream(stream)),
           "r4_prepack_blockfp8")


def r4_gemm_workspace_bytes(op, M, N, K):
    return int(lib().r4_gemm_workspace_bytes(op, M, N, K))


PLAN_FIELDS = ("token_tile", "weight_rows", "n_tiles", "t_tiles", "splits", "kb_per_split", "units", "grid",
               "cluster", "stream_k")


def r4_plan_gemm(op, M, N, K, sms):
    """The schedule a GEMM call would launch on `sms` SMs (host arithmetic),
    as a dict keyed by PLAN_FIELDS."""
    out = (ctypes.c_int32 * len(PLAN_FIELDS))()
    _check(lib().r4_plan_gemm(op, M, N, K, sms, ctypes.cast(out, ctypes.c_void_p)), "r4_plan_gemm")
    return dict(zip(PLAN_FIELDS, list(out)))


def _ws(workspace):
    if workspace is None:
        return None, 0
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def r4_gemm_w4a8_mxfp4(q, s, packed, M, N, K, c, ldc, workspace=None, stream=None):
    _need(q, torch.uint8, "q"); _need(s, torch.float32, "s"); _need(c, torch.bfloat16, "c")
    wp, wb = _ws(workspace)
    _check(lib().r4_gemm_w4a8_mxfp4(_ptr(q), _ptr(s), _ptr(packed), M, N, K, _ptr(c), ldc, wp, wb, _stream(stream)),
           "r4_gemm_w4a8_mxfp4")


def r4_linear_w4a8_mxfp4(x, ldx, packed, M, N, K, c, ldc, workspace, stream=None):
    _need(x, torch.bfloat16, "x"); _need(c, torch.bfloat16, "c")
    wp, wb = _ws(workspace)
    _check(lib().r4_linear_w4a8_mxfp4(_ptr(x), ldx, _ptr(packed), M, N, K, _ptr(c), ldc, wp, wb, _stream(stream)),
           "r4_linear_w4a8_mxfp4")


def r4_gemm_w4a8_mxfp4_noalloc(q, s, packed, M, N, K, c, ldc, stream=None):
    """W4A8 GEMM without a caller workspace (split-K scratch is the library's
    static device buffer); for callers that cannot allocate device memory."""
    _need(q, torch.uint8, "q"); _need(s, torch.float32, "s"); _need(c, torch.bfloat16, "c")
    _check(lib().r4_gemm_w4a8_mxfp4_noalloc(_ptr(q), _ptr(s), _ptr(packed), M, N, K, _ptr(c), ldc, _stream(stream)),
           "r4_gemm_w4a8_mxfp4_noalloc")


def r4_gemm_w4a4_mxfp4(q, q_scale, packed, M, N, K, c, ldc, workspace=None, stream=None):
    _need(q, torch.uint8, "q"); _need(q_scale, torch.uint8, "q_scale"); _need(c, torch.bfloat16, "c")
    wp, wb = _ws(workspace)
    _check(lib().r4_gemm_w4a4_mxfp4(_ptr(q), _ptr(q_scale), _ptr(packed), M, N, K, _ptr(c), ldc, wp, wb,
                                    _stream(stream)), "r4_gemm_w4a4_mxfp4")


def r4_gemm_blockfp8(q, As, packed, M, N, K, c, ldc, workspace=None, stream=None):
    _need(q, torch.uint8, "q"); _need(As, torch.float32, "As"); _need(c, torch.bfloat16, "c")
    wp, wb = _ws(workspace)
    _check(lib().r4_gemm_blockfp8(_ptr(q), _ptr(As), _ptr(packed), M, N, K, _ptr(c), ldc, wp, wb, _stream(stream)),
           "r4_gemm_blockfp8")


def r4_gemm_bf16_nt_skinny(x, w, M, N, K, c, ldc, workspace=None, stream=None):
    _need(x, torch.bfloat16, "x"); _need(w, torch.bfloat16, "w"); _need(c, torch.bfloat16, "c")
    wp, wb = _ws(workspace)
    _check(lib().r4_gemm_bf16_nt_skinny(_ptr(x), _ptr(w), M, N, K, _ptr(c), ldc, wp, wb, _stream(stream)),
           "r4_gemm_bf16_nt_skinny")


def r4_add_rmsnorm_quant_fp8(y, residual, weight, eps, M, K, residual_out, q, s, stream=None):
    _need(y, torch.bfloat16, "y"); _need(residual, torch.bfloat16, "residual")
    _need(weight, torch.bfloat16, "weight"); _need(residual_out, torch.bfloat16, "residual_out")
    _need(q, torch.uint8, "q"); _need(s, torch.float32, "s")
    _check(lib().r4_add_rmsnorm_quant_fp8(_ptr(y), _ptr(residual), _ptr(weight), float(eps), M, K,
                                          _ptr(residual_out), _ptr(q), _ptr(s), _stream(stream)),
           "r4_add_rmsnorm_quant_fp8")


def r4_check_quotients(count, example, stream=None):
    _need(count, torch.int64, "count"); _need(example, torch.float32, "example")
    _check(lib().r4_check_quotients(_ptr(count), _ptr(example), _stream(stream)), "r4_check_quotients")


def r4_mma_peak(kind, n, blocks, iters, stream=None):
    _check(lib().r4_mma_peak(int(kind), int(n), int(blocks), int(iters), _stream(stream)), "r4_mma_peak")


def r4_silu_mul_quant_fp8(gu, M, N, q, s, stream=None):
    _need(gu, torch.bfloat16, "gu"); _need(q, torch.uint8, "q"); _need(s, torch.float32, "s")
    _check(lib().r4_silu_mul_quant_fp8(_ptr(gu), M, N, _ptr(q), _ptr(s), _stream(stream)), "r4_silu_mul_quant_fp8")


# --------------------------------------------------------------------------- helpers

def quant_fp8(x, group=None, stream=None):
    """x bf16 [M, K] (row stride may exceed K) -> (q uint8 [M, K], s fp32 [M] or [M, K/128])."""
    M, K = x.shape
    assert x.stride(1) == 1
    g = K if group is None else group
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((M,) if group is None else (M, K // g), dtype=torch.float32, device=x.device)
    r4_quant_fp8_per_token(x, M, K, x.stride(0), g, q, s, stream)
    return q, s


def quant_mxfp4(x, stream=None):
    """x bf16 [M, K] (row stride may exceed K) -> (q uint8 [M, K/2] packed e2m1,
    scale uint8 atoms for r4_gemm_w4a4_mxfp4)."""
    M, K = x.shape
    assert x.stride(1) == 1
    q = torch.empty((M, K // 2), dtype=torch.uint8, device=x.device)
    sc = torch.empty(r4_quant_mxfp4_act_scale_bytes(M, K), dtype=torch.uint8, device=x.device)
    r4_quant_mxfp4_act(x, M, K, x.stride(0), q, sc, stream)
    return q, sc


def add_rmsnorm_quant(y, residual, weight, eps, residual_out=None, stream=None):
    """y, residual bf16 [M, K], weight bf16 [K] -> (q uint8 [M, K], s fp32 [M], residual_out bf16 [M, K]).
    Pass residual_out=residual for the in-place residual update."""
    M, K = y.shape
    assert y.is_contiguous() and residual.is_contiguous() and weight.is_contiguous()
    ro = torch.empty_like(residual) if residual_out is None else residual_out
    q = torch.empty((M, K), dtype=torch.uint8, device=y.device)
    s = torch.empty((M,), dtype=torch.float32, device=y.device)
    r4_add_rmsnorm_quant_fp8(y, residual, weight, eps, M, K, ro, q, s, stream)
    return q, s, ro


def silu_mul_quant(gu, stream=None):
    """gu bf16 [M, 2N] = [gate | up] -> (q uint8 [M, N], s fp32 [M])."""
    M, N2 = gu.shape
    assert gu.is_contiguous() and N2 % 2 == 0
    N = N2 // 2
    q = torch.empty((M, N), dtype=torch.uint8, device=gu.device)
    s = torch.empty((M,), dtype=torch.float32, device=gu.device)
    r4_silu_mul_quant_fp8(gu, M, N, q, s, stream)
    return q, s


def quantize_mxfp4_weight(w, stream=None):
    N, K = w.shape
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    scale = torch.empty((N, K // 32), dtype=torch.uint8, device=w.device)
    r4_quantize_mxfp4_weight(w.contiguous(), N, K, packed, scale, stream)
    return packed, scale


def quantize_blockfp8_weight(w, stream=None):
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    r4_quantize_blockfp8_weight(w.contiguous(), N, K, q, s, stream)
    return q, s


def prepack_mxfp4(w, w_scale, N, K, stream=None):
    packed = torch.empty(r4_prepack_mxfp4_bytes(N, K), dtype=torch.uint8, device=w.device)
    r4_prepack_mxfp4(w.contiguous(), w_scale.contiguous(), N, K, packed, stream)
    return packed


def prepack_blockfp8(w, w_scale, N, K, stream=None):
    packed = torch.empty(r4_prepack_blockfp8_bytes(N, K), dtype=torch.uint8, device=w.device)
    r4_prepack_blockfp8(w.contiguous(), w_scale.contiguous(), N, K, packed, stream)
    return packed


def workspace(op, M, N, K, device="cuda"):
    """Zeroed workspace for a GEMM call (None when the schedule needs none)."""
    n = r4_gemm_workspace_bytes(op, M, N, K)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device)


def linear_w4a8(x, packed, N, K, ws=None, out=None, stream=None):
    """bf16 activations x [M, K] (row stride x.stride(0)) -> bf16 [M, N]:
    per-token quantization and the W4A8 GEMM in one call."""
    M = x.shape[0]
    c = torch.empty((M, N), dtype=torch.bfloat16, device=x.device) if out is None else out
    if ws is None:
        ws = workspace(R4_OP_LINEAR_W4A8_MXFP4, M, N, K, x.device)
    r4_linear_w4a8_mxfp4(x, x.stride(0), packed, M, N, K, c, c.stride(0), ws, stream)
    return c


def gemm_w4a8(q, s, packed, N, K, ws=None, out=None, stream=None):
    M = q.shape[0]
    c = torch.empty((M, N), dtype=torch.bfloat16, device=q.device) if out is None else out
    if ws is None:
        ws = workspace(R4_OP_W4A8_MXFP4, M, N, K, q.device)
    r4_gemm_w4a8_mxfp4(q, s, packed, M, N, K, c, c.stride(0), ws, stream)
    return c


def gemm_w4a4(q, q_scale, packed, N, K, ws=None, out=None, stream=None):
    M = q.shape[0]
    c = torch.empty((M, N), dtype=torch.bfloat16, device=q.device) if out is None else out
    if ws is None:
        ws = workspace(R4_OP_W4A4_MXFP4, M, N, K, q.device)
    r4_gemm_w4a4_mxfp4(q, q_scale, packed, M, N, K, c, c.stride(0), ws, stream)
    return c


def gemm_blockfp8(q, As, packed, N, K, ws=None, out=None, stream=None):
    M = q.shape[0]
    c = torch.empty((M, N), dtype=torch.bfloat16, device=q.device) if out is None else out
    if ws is None:
        ws = workspace(R4_OP_BLOCKFP8, M, N, K, q.device)
    r4_gemm_blockfp8(q, As, packed, M, N, K, c, c.stride(0), ws, stream)
    return c


def gemm_bf16_skinny(x, w, out=None, stream=None):
    M, K = x.shape
    N = w.shape[0]
    c = torch.empty((M, N), dtype=torch.bfloat16, device=x.device) if out is None else out
    r4_gemm_bf16_nt_skinny(x.contiguous(), w.contiguous(), M, N, K, c, c.stride(0), None, stream)
    return c
