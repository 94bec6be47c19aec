"""Exact number formats used by the experts forward (oracle side, fp64).

Test infrastructure only (see the package docstring).

* e4m3 ("fn" variant, OCP 8-bit floating point): 1 sign, 4 exponent bits
  (bias 7), 3 mantissa bits, no infinities, codes 0x7F / 0xFF are NaN, largest
  finite magnitude 448.
* e2m1 (OCP microscaling FP4): 1 sign, 2 exponent bits (bias 1), 1 mantissa
  bit, no NaN/Inf; magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* UE8M0: an unsigned power-of-two exponent byte, value 2^(b-127); 0xFF is NaN.

The activation rule (1x128 blocks, power-of-two scale 2^ceil(log2(amax/448)),
e4m3 codes) is the "dynamic per-block" activation quantization that the
finegrained_fp8 page says the grouped experts dispatch performs; its exact
form comes from the workload definitions. Readings taken here:

* the exponent is the exact integer e = min{n : amax <= 448 * 2^n}, which is
  the formula above in exact arithmetic; amax = 0 gives e = 0; e is clamped to
  [-127, 127] so that it fits a UE8M0 byte;
* the conversion to e4m3 is round-to-nearest, ties to the even code, with
  saturation to +-448 (never reached by the rule above), and keeps the sign
  of zero (a negative value that rounds to zero gives 0x80);
* a partial last block (dim % 128 != 0) covers only the existing elements.

FP4 activations (the variant in which both GEMM operands are e2m1, the
FP4 x FP4 block-scaled MMA named next to the FP8 x FP4 one): the pages give
no activation rule for it, so the microscaling blocking of the FP4 weights is
taken: 1x32 blocks, one UE8M0 exponent per block, e2m1 codes. Readings:

* n = min{n : amax <= 6 * 2^n} (6 is the largest e2m1 magnitude), the same
  rule as for the FP4 weight data; amax = 0 gives n = 0; n is clamped to
  [-127, 127];
* the conversion to e2m1 is round-to-nearest, ties to the even code, with
  saturation to +-6 (never reached by the rule above), and keeps the sign of
  zero (a negative value that rounds to zero gives code 0x8);
* codes are packed two per byte with the even element in the low nibble, as
  for the FP4 weights.
"""
import numpy as np

E4M3_MAX = 448.0
ACT_BLOCK = 128
E2M1_MAX = 6.0
ACT_BLOCK_FP4 = 32


def _e4m3_value(code):
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * 2.0 ** -6 * (m / 8.0)
    return s * 2.0 ** (e - 7) * (1.0 + m / 8.0)


def _e2m1_value(code):
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * 0.5 * m
    return s * 2.0 ** (e - 1) * (1.0 + m / 2.0)


def _ue8m0_value(code):
    if code == 0xFF:
        return float("nan")
    return 2.0 ** (code - 127)


# Decode tables indexed by the raw code, built from the bit-field definitions.
E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)
UE8M0_TABLE = np.array([_ue8m0_value(c) for c in range(256)], dtype=np.float64)


def decode_e4m3(codes):
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def decode_e2m1_packed(packed, k):
    """Unpack int8/uint8 bytes holding two e2m1 codes each into fp64 values.

    Reading (the pages only say "FP4-packed in int8"): the low nibble holds
    the even element along K, the high nibble the odd one. ``k`` is the
    logical length of the last axis.
    """
    b = np.asarray(packed).view(np.uint8)
    lo = b & 0xF
    hi = b >> 4
    codes = np.empty(b.shape[:-1] + (b.shape[-1] * 2,), dtype=np.uint8)
    codes[..., 0::2] = lo
    codes[..., 1::2] = hi
    return E2M1_TABLE[codes[..., :k]]


def decode_ue8m0(codes):
    return UE8M0_TABLE[np.asarray(codes, dtype=np.uint8)]


# Positive finite e4m3 magnitudes in code order 0x00..0x7E (ascending).
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = E4M3_TABLE[:0x7F]


def e4m3_rne_satfinite(v):
    """Round fp64 values to e4m3 codes: nearest, ties to even code, saturate.

    The value set is searched directly: the two neighbouring magnitudes are
    compared and an exact tie goes to the code whose mantissa LSB is 0.
    """
    v = np.asarray(v, dtype=np.float64)
    if np.isnan(v).any():
        raise ValueError("NaN input to the e4m3 quantizer")
    mag = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, mag, side="left")  # first >= mag
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS_VALUES[hi] - mag
    d_lo = mag - _POS_VALUES[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((hi & 1) == 0))
    exact = _POS_VALUES[hi] == mag
    code = np.where(exact | pick_hi, hi, lo).astype(np.uint8)
    sign = np.signbit(v)
    return np.where(sign, code | 0x80, code).astype(np.uint8)


def act_scale_exponent(amax):
    """e = min{n : amax <= 448 * 2^n}, 0 for amax == 0, clamped to [-127, 127].

    With amax = m * 2^E (m in [0.5, 1), numpy.frexp) and 448 = 0.875 * 2^9:
    amax <= 0.875 * 2^(9+n)  <=>  n >= E - 9 when m <= 0.875, else n >= E - 8.
    """
    amax = np.asarray(amax, dtype=np.float64)
    m, E = np.frexp(amax)
    n = np.where(m <= 0.875, E - 9, E - 8)
    n = np.where(amax == 0, 0, n)
    return np.clip(n, -127, 127).astype(np.int32)


def quantize_rows_1x128(x):
    """Dynamic 1x128 activation quantization of a 2-D fp64 array.

    Returns (codes uint8 [R, D], exps int32 [R, ceil(D/128)]) with
    x ~= decode_e4m3(codes) * 2^exps (block-broadcast).
    """
    x = np.asarray(x, dtype=np.float64)
    R, D = x.shape
    nb = (D + ACT_BLOCK - 1) // ACT_BLOCK
    codes = np.empty((R, D), dtype=np.uint8)
    exps = np.empty((R, nb), dtype=np.int32)
    for b in range(nb):
        lo, hi = b * ACT_BLOCK, min(D, (b + 1) * ACT_BLOCK)
        blk = x[:, lo:hi]
        e = act_scale_exponent(np.max(np.abs(blk), axis=1))
        exps[:, b] = e
        codes[:, lo:hi] = e4m3_rne_satfinite(blk * np.ldexp(1.0, -e)[:, None])
    return codes, exps


def dequantize_rows_1x128(codes, exps):
    vals = decode_e4m3(codes)
    D = vals.shape[1]
    scale = np.repeat(np.ldexp(1.0, exps.astype(np.int64)), ACT_BLOCK, axis=1)[:, :D]
    return vals * scale


# Non-negative e2m1 magnitudes in code order 0..7 (ascending).
_E2M1_POS = E2M1_TABLE[:8]


def e2m1_rne_satfinite(v):
    """Round fp64 values to 4-bit e2m1 codes: nearest, ties to even code,
    saturate at 6; the sign bit (0x8) follows the sign of v, zero included."""
    v = np.asarray(v, dtype=np.float64)
    if np.isnan(v).any():
        raise ValueError("NaN input to the e2m1 quantizer")
    mag = np.minimum(np.abs(v), E2M1_MAX)
    hi = np.minimum(np.searchsorted(_E2M1_POS, mag, side="left"), 7)  # first >= mag
    lo = np.maximum(hi - 1, 0)
    d_hi = _E2M1_POS[hi] - mag
    d_lo = mag - _E2M1_POS[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((hi & 1) == 0))
    exact = _E2M1_POS[hi] == mag
    code = np.where(exact | pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(v), code | 0x8, code).astype(np.uint8)


def act_scale_exponent_e2m1(amax):
    """n = min{n : amax <= 6 * 2^n}, 0 for amax == 0, clamped to [-127, 127].

    With amax = m * 2^E (m in [0.5, 1), numpy.frexp) and 6 = 0.75 * 2^3:
    amax <= 0.75 * 2^(3+n)  <=>  n >= E - 3 when m <= 0.75, else n >= E - 2.
    """
    amax = np.asarray(amax, dtype=np.float64)
    m, E = np.frexp(amax)
    n = np.where(m <= 0.75, E - 3, E - 2)
    n = np.where(amax == 0, 0, n)
    return np.clip(n, -127, 127).astype(np.int32)


def quantize_rows_1x32_e2m1(x):
    """Dynamic 1x32 FP4 activation quantization of a 2-D fp64 array.

    Returns (codes uint8 [R, D], one 4-bit code per element, and exps int32
    [R, ceil(D/32)]) with x ~= E2M1_TABLE[codes] * 2^exps (block-broadcast).
    """
    x = np.asarray(x, dtype=np.float64)
    R, D = x.shape
    nb = (D + ACT_BLOCK_FP4 - 1) // ACT_BLOCK_FP4
    codes = np.empty((R, D), dtype=np.uint8)
    exps = np.empty((R, nb), dtype=np.int32)
    for b in range(nb):
        lo, hi = b * ACT_BLOCK_FP4, min(D, (b + 1) * ACT_BLOCK_FP4)
        blk = x[:, lo:hi]
        e = act_scale_exponent_e2m1(np.max(np.abs(blk), axis=1))
        exps[:, b] = e
        codes[:, lo:hi] = e2m1_rne_satfinite(blk * np.ldexp(1.0, -e)[:, None])
    return codes, exps


def dequantize_rows_1x32_e2m1(codes, exps):
    vals = E2M1_TABLE[np.asarray(codes, dtype=np.uint8)]
    D = vals.shape[1]
    scale = np.repeat(np.ldexp(1.0, exps.astype(np.int64)), ACT_BLOCK_FP4, axis=1)[:, :D]
    return vals * scale


def pack_e2m1(codes):
    """4-bit codes [R, D] (D even) -> bytes [R, D/2], even element in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def bf16_bits_to_f64(bits):
    """bf16 bit patterns (uint16) -> fp64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):  # NaN patterns stay NaN (no warning)
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16_rne(v):
    """fp64 -> nearest bf16 value (ties to even), returned as fp64.

    bf16 keeps 8 significant bits: with |v| = m * 2^E (m in [0.5, 1)) the
    spacing is 2^(E-8), or 2^-133 in the subnormal range. numpy.round rounds
    halves to even. Used only to report errors against a bf16-rounded oracle.
    """
    v = np.asarray(v, dtype=np.float64)
    _, E = np.frexp(v)
    ulp = np.ldexp(1.0, np.maximum(E - 8, -133))
    return np.round(v / ulp) * ulp
