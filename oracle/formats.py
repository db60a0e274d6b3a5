"""Number formats used by the oracle: BF16 and FP8 E4M3 ("e4m3fn"), written from their
format definitions.  Test infrastructure only (see the package docstring).

BF16: 1 sign bit, 8 exponent bits (bias 127), 7 stored mantissa bits -- the top half
of an IEEE float32.  Conversion from float32 rounds to nearest, ties to even.

E4M3 (the "fn" variant used by the FP8 dispatch of the DeepEP page and by the combine
fake-quant of the Mega-MoE page): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits,
no infinities.  Exponent field 0 holds subnormals m * 2^-9; exponent field 15 with
mantissa 7 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.  Encoding rounds
to nearest, ties to even, and saturates finite values beyond 448 to +-448 ("satfinite").

E2M1 (the element format of NVFP4, the 4-bit combine and dispatch units the Mega-MoE page
names next to the FP8 ones): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no
infinities or NaN.  Exponent field 0 holds the subnormal 0.5 * m, so the magnitudes are
0, 0.5, 1, 1.5, 2, 3, 4 and 6.  Encoding rounds to nearest, ties to even, and saturates
beyond 6.

Pinned in tests/test_oracle_formats.py against torch's CPU casts (library routines) on
exhaustive or large seeded sets, and against the definition's special cases; E2M1 in
tests/test_oracle_nvfp4.py against its value table and a brute-force nearest search.
"""
import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_SUBNORMAL_STEP = 2.0 ** -9


def f32_to_bf16_bits(x):
    """float32 array -> uint16 BF16 bit patterns, round to nearest even.

    The 16 discarded low bits are compared with the halfway point 0x8000; above it, or
    at it with an odd kept part, the kept part is incremented (a carry into the
    exponent is the correct result, including overflow to infinity).  NaN stays NaN.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    kept = u >> 16
    low = u & 0xFFFF
    up = (low > 0x8000) | ((low == 0x8000) & ((kept & 1) == 1))
    out = (kept + up.astype(np.uint64)).astype(np.uint32)
    nan = np.isnan(x)
    out = np.where(nan, (kept & 0x8000) | 0x7FC0, out)
    return out.astype(np.uint16)


def bf16_bits_to_f32(b):
    """uint16 BF16 bit patterns -> float32 (exact)."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_round(x):
    """float32 -> nearest-even BF16 value, returned as float32."""
    return bf16_bits_to_f32(f32_to_bf16_bits(x))


def _e4m3_value(c):
    """Value of E4M3 codes (int64 array) from the format definition."""
    sign = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    man = c & 0x7
    sub = man * E4M3_SUBNORMAL_STEP
    norm = (1.0 + man / 8.0) * np.exp2(ex - 7.0)
    mag = np.where(ex == 0, sub, norm)
    mag = np.where((ex == 15) & (man == 7), np.nan, mag)
    return (sign * mag).astype(np.float32)


# the value of every one of the 256 codes, from the definition above
_E4M3_TABLE = _e4m3_value(np.arange(256, dtype=np.int64))
_E4M3_TABLE64 = _E4M3_TABLE.astype(np.float64)


def e4m3_decode(codes):
    """uint8 E4M3 codes -> float32 values (exact); codes 0x7F / 0xFF decode to NaN.
    A lookup in the table of all 256 code values."""
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_decode64(codes):
    """e4m3_decode, as float64 (exact: every E4M3 value is a float32 and a float64)."""
    return _E4M3_TABLE64[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x):
    """float32 array -> uint8 E4M3 codes: round to nearest even, saturate to +-448.

    Read off the float32 bit pattern.  At or above the smallest normal 2^-6, E4M3 keeps 3
    of float32's 23 fraction bits: the 20 dropped bits are rounded to nearest, ties to
    even (adding 0x7FFFF plus the lowest kept bit, then shifting; a carry moves into the
    exponent, which is the correctly rounded result), and the exponent is rebiased from
    127 to 7, i.e. the code is the shifted pattern minus (127 - 7) << 3.  Below 2^-6 the
    values are the multiples m * 2^-9 (m = 0..8, 8 being 2^-6 itself), so the code is
    |x| * 2^9 rounded half to even.  Codes past 126 (448) saturate to 126; NaN gives
    0x7F.  The sign bit is copied.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    mag = u & np.uint32(0x7FFFFFFF)
    small = mag < np.uint32(0x3C800000)                          # below 2^-6
    nan = mag > np.uint32(0x7F800000)
    # normal range: round the dropped 20 bits to nearest even, then rebias the exponent
    code = mag >> np.uint32(20)
    code &= np.uint32(1)
    code += mag
    code += np.uint32(0x7FFFF)
    code >>= np.uint32(20)
    code = code.view(np.int32)
    code -= np.int32((127 - 7) << 3)
    # subnormal range: |x| * 2^9 rounded half to even (computed for every element, used only
    # where |x| < 2^-6; the others may overflow or be NaN, harmlessly)
    with np.errstate(over="ignore", invalid="ignore"):
        sub = np.abs(x)
        sub *= np.float32(512.0)
        np.rint(sub, out=sub)
        np.copyto(code, sub.astype(np.int32), where=small)
    np.minimum(code, np.int32(0x7E), out=code)
    code[nan] = 0x7F
    code |= ((u >> np.uint32(24)) & np.uint32(0x80)).view(np.int32)
    return code.astype(np.uint8)


def e4m3_round(x):
    """float32 -> nearest-even, saturated E4M3 value, returned as float32."""
    return e4m3_decode(e4m3_encode(x))


E2M1_MAX = 6.0


def e2m1_decode(codes):
    """uint8 E2M1 codes (low 4 bits) -> float32 values (exact)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    ex = (c >> 1) & 0x3
    man = c & 0x1
    mag = np.where(ex == 0, 0.5 * man, (1.0 + 0.5 * man) * np.exp2(ex - 1.0))
    return (sign * mag).astype(np.float32)


def e2m1_encode(x):
    """float32 array -> uint8 E2M1 codes: round to nearest even, saturate to +-6.

    As for E4M3: in float64, the spacing of E2M1 values around |x| is 0.5 below 2 (the
    subnormal step, which the first binade [1, 2) shares), else 2^(e-1) for
    2^e <= |x| < 2^(e+1); |x| / spacing is rounded half to even and scaled back, clamped
    to 6, and the code read off the rounded value.  NaN inputs are not defined for the
    format and are not expected."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    _, ex = np.frexp(a)
    e = ex.astype(np.int64) - 1
    step = np.where(a < 2.0, 0.5, np.exp2(np.maximum(e, 1) - 1.0))
    v = np.minimum(np.rint(a / step) * step, E2M1_MAX)
    # codes: 0 0.5 1 1.5 2 3 4 6 -> 0..7
    mag_code = np.where(v < 2.0, np.rint(v / 0.5), np.where(v < 4.0, 2 + v, 4 + v / 2.0)).astype(np.int64)
    return (mag_code | np.where(neg, 0x8, 0)).astype(np.uint8)


def e2m1_round(x):
    """float32 -> nearest-even, saturated E2M1 value, returned as float32."""
    return e2m1_decode(e2m1_encode(x))


def round_up(x, y):
    """Smallest multiple of y that is >= x (the tile-count helper of the DeepEP page)."""
    return ((x + y - 1) // y) * y
