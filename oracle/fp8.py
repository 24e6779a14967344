"""FP8 E4M3 keys of the k8v4 layer format (test infrastructure: the oracle).

[P1] §プリセット lists a preset that keeps the keys in FP8 and the values in
4-bit TurboQuant codes (k8v4), because the error of the method comes almost
entirely from the keys.  The pages do not spell the FP8 format out; the
reading (fixed in include/tq.h) is the E4M3 encoding NVIDIA GPUs convert to:

* 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
  holds subnormals m * 2^-9 (m = 1..7); no infinities; S.1111.111 is NaN, so
  the largest finite magnitude is 1.75 * 2^8 = 448;
* encoding rounds to nearest with ties to even, and saturates: a finite
  magnitude that rounds above 448 (and an infinity) becomes +-448; NaN stays NaN;
* keys are stored as the FP8 encoding of each raw key coordinate (no rotation,
  no scale): 128 bytes per token, 16 tokens per page, nothing else in the page.

Both functions work from that definition in float64 arithmetic, element by
element; they share nothing with the CUDA path.

Pinned by tests/test_oracle_fp8.py: every one of the 254 finite codes decodes
and re-encodes to itself, printed values of the format (1.0 = 0x38, 448 =
0x7E, 2^-6 = 0x08, 2^-9 = 0x01), ties to even at grid midpoints, saturation,
and agreement with PyTorch's float8_e4m3fn conversion on in-range values.
"""

import math

import numpy as np

MAX = 448.0
NAN_CODE = 0x7F


def decode_byte(b):
    """float value of one E4M3 byte (NaN for 0x7F / 0xFF)."""
    b = int(b) & 0xFF
    sign = -1.0 if b & 0x80 else 1.0
    e = (b >> 3) & 0xF
    m = b & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def _round_half_even(x):
    f = math.floor(x)
    r = x - f
    if r > 0.5:
        return f + 1
    if r < 0.5:
        return f
    return f if f % 2 == 0 else f + 1


def encode_value(x):
    """E4M3 byte of one real value: nearest, ties to even, saturating at +-448."""
    x = float(x)
    if math.isnan(x):
        return NAN_CODE
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    if math.isinf(a):
        return sign | 0x7E
    if a >= 2.0 ** -6:
        e = math.floor(math.log2(a))
        while 2.0 ** e > a:  # exact exponent despite log2 rounding
            e -= 1
        while 2.0 ** (e + 1) <= a:
            e += 1
        if e > 8:
            return sign | 0x7E
        q = _round_half_even((a / 2.0 ** e - 1.0) * 8.0)
        if q == 8:
            e, q = e + 1, 0
        if e > 8 or (e == 8 and q == 7):  # above 448: saturate
            return sign | 0x7E
        return sign | ((e + 7) << 3) | q
    q = _round_half_even(a / 2.0 ** -9)  # subnormal grid; q = 8 is 2^-6, code 0x08
    return sign | q


def encode(x):
    """Elementwise E4M3 bytes (uint8) of an array."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    flat = out.reshape(-1)
    for i, v in enumerate(x.reshape(-1)):
        flat[i] = encode_value(v)
    return out


_TABLE = np.array([decode_byte(b) for b in range(256)], dtype=np.float64)


def decode(b):
    """Elementwise float64 values of E4M3 bytes."""
    return _TABLE[np.asarray(b, dtype=np.uint8)]


def page_bytes(d):
    """Bytes of one key page of the k8v4 format (16 records of d bytes)."""
    return 16 * d
