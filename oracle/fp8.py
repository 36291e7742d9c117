"""FP8-E4M3 codec for the T2 (8-bit) tier.  Test infrastructure (see package doc).

Source of the method: the gist.science summary of "Not All Thoughts Need HBM",
section "Four-tier classification", item T2 (low-importance tokens kept at low
precision, e.g. 8-bit), and the ARKV summary, "Tri-state cache assignment"
(quantised tokens are dequantised on the fly before attention).  The pages fix
"8-bit" but no format; the format used is OCP FP8 E4M3 (the "fn" variant):

  * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
  * exponent field 0 encodes subnormals  (-1)^s * 2^-6 * (m / 8);
  * exponent fields 1..15 encode normals (-1)^s * 2^(e-7) * (1 + m / 8);
  * there are no infinities; S.1111.111 is NaN, so the largest finite
    magnitude is 0x7E = 2^8 * 1.75 = 448.

Per-row scaling (one fp32 scale per token, per layer, per KV head, separately
for K and V):

  scale = amax / 448            (fp32 division, IEEE round-to-nearest)
  y_j   = x_j / scale           (fp32 division, IEEE round-to-nearest)
  code  = nearest E4M3 value to y_j, ties to the even code, |y| > 448 -> 448
  x_j'  = value(code) * scale   (exact in fp64)

An all-zero row gets scale = 1 and all-zero codes.  The fp32 steps are taken in
fp32 on purpose: the quantised code is an integer decided by floating point,
so both this oracle and the GPU take that decision in the same precision.
"""

import numpy as np

E4M3_MAX = 448.0
NAN_CODES = (0x7F, 0xFF)


def decode(code: int) -> float:
    """Value of one E4M3 code, from the bit fields (NaN for S.1111.111)."""
    code = int(code) & 0xFF
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp_field = (code >> 3) & 0xF
    mant = code & 0x7
    if exp_field == 0xF and mant == 0x7:
        return float("nan")
    if exp_field == 0:
        return sign * (2.0 ** -6) * (mant / 8.0)
    return sign * (2.0 ** (exp_field - 7)) * (1.0 + mant / 8.0)


# Value of every code, in code order.
DECODE_TABLE = np.array([decode(c) for c in range(256)], dtype=np.float64)

# Non-negative finite magnitudes: codes 0x00..0x7E, strictly increasing.
_POS_VALUES = DECODE_TABLE[:0x7F].copy()


def encode(y) -> np.ndarray:
    """Round fp32 values to E4M3 codes: nearest value, ties to even, saturating.

    The search is over the table of finite non-negative values; the sign is
    taken from the sign bit of y (so -0.0 -> 0x80).  Ties between two adjacent
    codes go to the even code, which is the one whose mantissa LSB is 0.
    Magnitudes above 448 saturate to 448 (code 0x7E) -- "satfinite".
    Input must be finite.
    """
    y = np.asarray(y, dtype=np.float32)
    if not np.all(np.isfinite(y)):
        raise ValueError("E4M3 encode: input must be finite")
    mag = np.abs(y).astype(np.float64)
    neg = np.signbit(y)
    # index of the first table value >= mag
    hi = np.searchsorted(_POS_VALUES, mag, side="left")
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(mag >= E4M3_MAX, 0x7E, code)
    code = code.astype(np.uint8) | (neg.astype(np.uint8) << 7)
    return code


def quantise_row(x):
    """Quantise one row (a d-vector of bf16-exact values) -> (codes uint8[d], scale float32)."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0.0)
    if amax == 0.0:
        return np.zeros(x32.shape, dtype=np.uint8), np.float32(1.0)
    scale = np.float32(amax / np.float32(E4M3_MAX))
    y = (x32 / scale).astype(np.float32)
    return encode(y), scale


def dequantise_row(codes, scale) -> np.ndarray:
    """fp64 value of a quantised row: value(code) * scale."""
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8)] * np.float64(np.float32(scale))
