"""Number formats: decode tables and RNE encoders (oracle; test infrastructure only).

Every encoder here works by searching the sorted table of representable
magnitudes, never by bit manipulation, so that it cannot share a mistake with
a bit-twiddling implementation.

Formats
-------
e2m1 (OCP MX FP4): 1 sign, 2 exponent, 1 mantissa bit. The value table is the
    one printed on the radiance_mxfp4.py page in ``_exact_ref``:
    codes 0..15 -> [0, .5, 1, 1.5, 2, 3, 4, 6, -0, -.5, -1, -1.5, -2, -3, -4, -6].
e4m3 (OCP FP8 E4M3, "fn" variant, as torch.float8_e4m3fn used by
    ``_traced_quant`` on the radiance_mxfp4.py page): bias 7, no infinities,
    S.1111.111 is NaN, largest finite magnitude 448.
ue8m0 (OCP MX scale): an unsigned biased exponent, value 2^(code-127); the
    radiance_mxfp4.py page decodes it as ``pow(2, scale - 127)`` in
    ``_exact_ref``. Code 255 is NaN in the OCP MX specification.
bfloat16: 8 significant bits, float32 exponent range. All GEMMs round their
    float64 result to bfloat16 once, round-to-nearest-even.
"""

import numpy as np

# --- e2m1 -------------------------------------------------------------------

# radiance_mxfp4.py, ``_exact_ref``: the decode table, code -> value.
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                        -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0],
                       dtype=np.float64)
E2M1_MAX = 6.0


def e2m1_decode(codes):
    """e2m1 codes (0..15, any integer array) -> float64 values."""
    return E2M1_VALUES[np.asarray(codes, dtype=np.int64)]


def unpack_e2m1(packed, K):
    """[R, K/2] bytes -> [R, K] e2m1 codes.

    radiance_mxfp4.py, ``_exact_ref``: element 2j sits in the low nibble of
    byte j and element 2j+1 in its high nibble.
    """
    packed = np.asarray(packed, dtype=np.uint8)
    lo = packed & 0x0F
    hi = (packed >> 4) & 0x0F
    out = np.stack([lo, hi], axis=-1).reshape(packed.shape[0], K)
    return out


def pack_e2m1(codes):
    """[R, K] e2m1 codes -> [R, K/2] bytes (low nibble = even k)."""
    codes = np.asarray(codes, dtype=np.uint8)
    R, K = codes.shape
    assert K % 2 == 0
    c = codes.reshape(R, K // 2, 2)
    return (c[..., 0] | (c[..., 1] << 4)).astype(np.uint8)


def _rne_search(mag, table):
    """Index into the ascending ``table`` of the value nearest to each ``mag``.

    Ties go to the even index. For e2m1 and e4m3 the positive codes are the
    table indices themselves, and an even code has a zero mantissa LSB, so this
    is round-half-to-even in the format's own sense. ``mag`` beyond the last
    entry maps to the last entry (saturation).
    """
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.searchsorted(table, mag, side="left")
    hi = np.clip(hi, 0, len(table) - 1)
    lo = np.clip(hi - 1, 0, len(table) - 1)
    d_lo = np.abs(mag - table[lo])
    d_hi = np.abs(table[hi] - mag)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(mag >= table[-1], len(table) - 1, idx)
    return idx.astype(np.int64)


_E2M1_POS = E2M1_VALUES[:8]  # ascending 0, .5, ..., 6; index == code


def e2m1_encode_rne_sat(v):
    """float values -> e2m1 codes, round to nearest (ties to even), saturate at 6.

    The sign bit follows the sign of the input, so -0.0 and negatives that round
    to zero give code 8 (negative zero), as IEEE-style conversion does.
    """
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("e2m1 encoder: non-finite input")
    idx = _rne_search(np.abs(v), _E2M1_POS)
    sign = np.signbit(v).astype(np.int64) << 3
    return (idx | sign).astype(np.uint8)


# --- e4m3 -------------------------------------------------------------------

def _e4m3_closed_form(code):
    """Value of one e4m3 code by the OCP FP8 E4M3 definition."""
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        mag = (m / 8.0) * 2.0 ** (-6)
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


E4M3_VALUES = np.array([_e4m3_closed_form(c) for c in range(256)], dtype=np.float64)
E4M3_MAX = 448.0
_E4M3_POS = E4M3_VALUES[:0x7F]  # codes 0x00..0x7E, ascending, index == code


def e4m3_decode(codes):
    """e4m3 codes (uint8 array) -> float64 values (NaN for 0x7F / 0xFF)."""
    return E4M3_VALUES[np.asarray(codes, dtype=np.int64)]


def e4m3_encode_rne_sat(v):
    """float values -> e4m3 codes; RNE, finite values beyond 448 saturate to 448.

    Sign follows the input's sign bit (-0.0 -> 0x80). Non-finite input raises:
    the method leaves it unspecified (a NaN poisons the whole row's scale).
    """
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("e4m3 encoder: non-finite input")
    idx = _rne_search(np.abs(v), _E4M3_POS)
    sign = np.signbit(v).astype(np.int64) << 7
    return (idx | sign).astype(np.uint8)


# --- ue8m0 ------------------------------------------------------------------

def ue8m0_decode(codes):
    """ue8m0 scale codes -> float64 2^(code-127); code 255 -> NaN."""
    c = np.asarray(codes, dtype=np.int64)
    out = np.ldexp(1.0, c - 127)
    return np.where(c == 255, np.nan, out)


# --- bfloat16 ---------------------------------------------------------------

BF16_MAX = float(np.ldexp(255.0, 120))  # (2 - 2^-7) * 2^127


def bf16_round(v):
    """float64 -> nearest bfloat16 value (ties to even), returned as float64.

    One rounding straight from float64: the value is scaled by the power of two
    that puts the bfloat16 quantum at 1, rounded with np.rint (half to even),
    and scaled back. Subnormal quantum 2^-133; magnitudes that round past the
    largest finite bfloat16 become infinity.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.array(v, copy=True)
    finite = np.isfinite(v) & (v != 0)
    _, e = np.frexp(v[finite])              # |v| = m 2^e, 0.5 <= m < 1
    q = np.maximum(e - 8, -133)             # quantum exponent: 8 significant bits
    r = np.rint(np.ldexp(v[finite], -q))
    res = np.ldexp(r, q)
    res = np.where(np.abs(res) > BF16_MAX, np.copysign(np.inf, res), res)
    out[finite] = res
    return out


def bf16_bits(v):
    """bfloat16-representable float64 values -> uint16 bit patterns."""
    f32 = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f32.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(bits):
    """uint16 bfloat16 bit patterns -> float64 values."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)
