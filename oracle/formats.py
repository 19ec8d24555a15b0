"""Number formats of the block-FP8 MoE layer, written out from their definitions.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module; only
the tests, the smoke check and the CPU-baseline leg of the benchmark do.

Formats (all three pages use them; the vLLM "Skip padded work in block-FP8
DeepGemmExperts" page, section Purpose, names the FP8 E4M3 weights with
128x128 scales and the packed UE8M0 activation scales):

* FP8 E4M3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
  bits, no infinities, the all-ones pattern S.1111.111 is NaN, the largest
  finite magnitude is 448.  Exponent field 0 encodes subnormals m/8 * 2^-6.
* BF16: the upper 16 bits of an IEEE fp32; conversion is round-to-nearest-even.
* UE8M0: an unsigned 8-bit biased exponent b standing for 2^(b-127).
* fp32 fused multiply-add: a*b + c with a single rounding.

Every function takes and returns numpy arrays.
"""

import numpy as np

E4M3_MAX = 448.0
E4M3_NAN_CODE = 0x7F


def e4m3_decode_table() -> np.ndarray:
    """Value of each of the 256 E4M3 codes, as float64 (NaN for the two NaN codes)."""
    vals = np.empty(256, np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp_field = (code >> 3) & 0xF
        mant = code & 0x7
        if exp_field == 0xF and mant == 0x7:
            vals[code] = np.nan
        elif exp_field == 0:
            vals[code] = sign * (mant / 8.0) * 2.0 ** -6
        else:
            vals[code] = sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)
    return vals


E4M3_VALUES = e4m3_decode_table()
# codes 0x00..0x7E are the non-negative finite values in increasing order
_POS_VALUES = E4M3_VALUES[:0x7F].copy()
_MIDPOINTS = (_POS_VALUES[:-1] + _POS_VALUES[1:]) / 2.0  # 126 midpoints, exact in f64


def e4m3_decode(codes) -> np.ndarray:
    """uint8 codes -> float64 values."""
    return E4M3_VALUES[np.asarray(codes, np.uint8)]


def e4m3_encode(v) -> np.ndarray:
    """fp32 -> E4M3 codes, round to nearest with ties to the even code, saturating.

    Magnitudes past the largest finite value saturate to +-448 (the 'satfinite'
    behaviour); the sign of a result that rounds to zero is kept (-0 is 0x80);
    NaN maps to 0x7F.
    """
    v = np.asarray(v, np.float32)
    mag = np.abs(v).astype(np.float64)
    # i = number of midpoints strictly below mag: MID[i-1] < mag <= MID[i]
    idx = np.searchsorted(_MIDPOINTS, mag, side="left")
    clipped = np.minimum(idx, _MIDPOINTS.size - 1)
    on_tie = (idx < _MIDPOINTS.size) & (mag == _MIDPOINTS[clipped])
    # on a tie between codes i and i+1 take the even one
    code = np.where(on_tie & (idx % 2 == 1), idx + 1, idx)
    code = np.minimum(code, 0x7E).astype(np.uint8)  # saturate to 448
    code = np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(v), np.uint8(E4M3_NAN_CODE), code).astype(np.uint8)


def bf16_round(x) -> np.ndarray:
    """fp32 -> nearest BF16 (ties to even), returned as fp32 holding the BF16 value."""
    x = np.asarray(x, np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = (((bits + 0x7FFF + lsb) >> 16) << 16).astype(np.uint32)
    out = rounded.view(np.float32)
    return np.where(np.isnan(x), np.float32(np.nan), out).astype(np.float32)


def bf16_bits(x) -> np.ndarray:
    """fp32 holding a BF16 value -> its 16-bit pattern."""
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(bits) -> np.ndarray:
    """16-bit BF16 patterns -> fp32 values."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def ue8m0_to_f32(b) -> np.ndarray:
    """UE8M0 byte b -> 2^(b-127) as fp32 (exact; b in 1..254)."""
    b = np.asarray(b, np.uint8).astype(np.uint32)
    return (b << 23).view(np.float32)


def pow2_ceil(s) -> np.ndarray:
    """Smallest power of two >= s, for positive normal fp32 s (exact).

    A positive normal fp32 is already a power of two exactly when its mantissa
    field is zero; otherwise the next power of two up has exponent field + 1
    and a zero mantissa.
    """
    bits = np.asarray(s, np.float32).view(np.uint32)
    exp_field = (bits >> 23) & 0xFF
    bump = (bits & 0x7FFFFF) != 0
    exp_field = exp_field + bump.astype(np.uint32)
    return (exp_field << 23).astype(np.uint32).view(np.float32)


def f32_exponent_field(s) -> np.ndarray:
    """Biased exponent field of positive fp32 values (the UE8M0 byte of a power of two)."""
    return ((np.asarray(s, np.float32).view(np.uint32) >> 23) & 0xFF).astype(np.uint8)


def fma_f32(a, b, c) -> np.ndarray:
    """a*b + c in fp32 with one rounding (round to nearest even).

    The product of two fp32 values is exact in float64 (48 significant bits).
    The sum with c is formed in float64 rounded to odd (TwoSum recovers the
    exact error; an inexact result with an even last bit is moved to its odd
    neighbour on the side of the exact value), and a float64 rounded to odd
    rounds correctly to fp32 because float64 carries more than 24+1 bits
    (S. Boldo, G. Melquiond, "Emulation of FMA and correctly rounded sums:
    proved algorithms using rounding to odd", IEEE Trans. Computers 2008).
    """
    a64 = np.asarray(a, np.float32).astype(np.float64)
    b64 = np.asarray(b, np.float32).astype(np.float64)
    c64 = np.asarray(c, np.float32).astype(np.float64)
    prod = a64 * b64
    s = prod + c64
    bb = s - prod
    err = (prod - (s - bb)) + (c64 - bb)
    s_bits = s.view(np.uint64)
    even = (s_bits & 1) == 0
    fix = (err != 0) & even & np.isfinite(s)
    toward = np.where(err > 0, np.inf, -np.inf)
    s_odd = np.where(fix, np.nextafter(s, toward), s)
    return s_odd.astype(np.float32)
