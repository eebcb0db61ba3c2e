"""Number formats read and written by the oracle (test infrastructure).

bf16: 1 sign, 8 exponent (bias 127), 7 mantissa bits -- the top half of an
IEEE binary32.  e4m3 (OCP FP8 "E4M3FN"): bias 7, subnormals, no infinities,
S.1111.111 is NaN.  e2m1 (OCP FP4): bias 1, one mantissa bit, no NaN/inf.
NVFP4 stores e2m1 values with one e4m3 scale per 16 consecutive elements; the
pages put the indexer's arithmetic in FP4 ([HYBRID]) and that the global KV cache is
kept in FP4 ([V41]).
"""
import numpy as np


def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 to bf16, to nearest with ties to even; returns uint16.

    Written for finite values in bf16's normal range (all this path produces):
    the significand is scaled to 8 bits, rounded with numpy's half-to-even
    rint, and the exactly representable result is read back as bits.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m * 2**e, 0.5 <= |m| < 1
    r = np.rint(m * 256.0)                  # 8 significant bits
    v = np.ldexp(r, e - 8).astype(np.float32)  # exact: v is on the bf16 grid
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def round_bf16(x) -> np.ndarray:
    """float64 -> nearest bf16 (ties to even) -> float64."""
    return bf16_to_f64(f64_to_bf16_bits(x))


def e2m1_value(code) -> np.ndarray:
    """Value of 4-bit e2m1 codes: sign bit 3, exponent bits 2..1, mantissa bit 0."""
    c = np.asarray(code, dtype=np.int64)
    sign = np.where(c & 8, -1.0, 1.0)
    e = (c >> 1) & 3
    mant = (c & 1).astype(np.float64)
    sub = mant * 0.5                                    # 2^(1-bias) * mant/2
    nrm = np.ldexp(1.0 + mant / 2.0, (e - 1).astype(np.int64))
    return sign * np.where(e == 0, sub, nrm)


def e4m3_value(byte) -> np.ndarray:
    """Value of e4m3 (E4M3FN) bytes; NaN for exponent 15 with mantissa 7."""
    b = np.asarray(byte, dtype=np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 15
    mant = (b & 7).astype(np.float64)
    sub = np.ldexp(mant / 8.0, -6)
    nrm = np.ldexp(1.0 + mant / 8.0, (e - 7).astype(np.int64))
    v = sign * np.where(e == 0, sub, nrm)
    return np.where((e == 15) & ((b & 7) == 7), np.nan, v)


def nvfp4_decode(packed, scale) -> np.ndarray:
    """NVFP4 rows -> float64.

    packed: uint8 [..., D/2], element 2i in the low nibble of byte i (reading R7);
    scale:  uint8 [..., D/16], the e4m3 scale of elements 16g .. 16g+15.
    """
    p = np.asarray(packed, dtype=np.uint8)
    s = np.asarray(scale, dtype=np.uint8)
    lo = e2m1_value(p & 0x0F)
    hi = e2m1_value(p >> 4)
    vals = np.stack([lo, hi], axis=-1).reshape(*p.shape[:-1], p.shape[-1] * 2)
    sc = np.repeat(e4m3_value(s), 16, axis=-1)
    return vals * sc


# ---------------------------------------------------------------------------
# NVFP4 quantisation of the indexer query ([HYBRID]: the lightning indexer
# computes in FP4; reading R16)
# ---------------------------------------------------------------------------
E2M1_MAGNITUDES = e2m1_value(np.arange(8))      # codes 0..7: 0, .5, 1, 1.5, 2, 3, 4, 6
E4M3_NONNEGATIVE = e4m3_value(np.arange(127))   # codes 0..126: 0 .. 448 (127 is NaN)


def nearest_code(y, table) -> np.ndarray:
    """Code of the table value nearest to each y (table ascending).

    Found by measuring the distance to every table value.  When two values
    are equally near (they are neighbours, one with an even code and one with
    an odd code) the even code wins: round to nearest, ties to even mantissa.
    A y beyond the last value gets the last code (saturation).
    """
    table = np.asarray(table, np.float64)
    # beyond the last value the last code is nearest; clamping first keeps a
    # huge y from making every distance round to the same number
    y = np.minimum(np.asarray(y, np.float64), table[-1])
    d = np.abs(y[..., None] - table)
    hit = d == d.min(axis=-1, keepdims=True)
    even = hit & (np.arange(len(table)) % 2 == 0)
    return np.where(even.any(axis=-1), even.argmax(axis=-1), hit.argmax(axis=-1))


def nvfp4_quantize(x):
    """fp64 [..., D] (D % 16 == 0) -> NVFP4 (packed uint8 [..., D/2], scale uint8 [..., D/16]).

    Reading R16, the rule of R7's keys applied to the indexer query: the
    scale of each group of 16 is the e4m3 value nearest to amax/6 (ties to
    even, saturating at 448); every element becomes the e2m1 value nearest to
    x/scale (ties to even, saturating at 6), sign kept, a zero magnitude
    stored as +0; a zero scale stores all-zero codes.  These decisions are
    exact in fp64 and in fp32 alike: for bf16 inputs, amax/6 and x/scale are
    never within 2^-9 (relative) of a rounding boundary unless they lie on it.
    """
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    assert D % 16 == 0
    g = x.reshape(*x.shape[:-1], D // 16, 16)
    amax = np.abs(g).max(axis=-1)
    sc = nearest_code(amax / 6.0, E4M3_NONNEGATIVE)
    s = E4M3_NONNEGATIVE[sc]
    y = np.abs(g) / np.where(s > 0, s, 1.0)[..., None]
    mag = np.where(s[..., None] > 0, nearest_code(y, E2M1_MAGNITUDES), 0)
    code = mag | np.where((g < 0) & (mag > 0), 8, 0)
    code = code.reshape(*x.shape[:-1], D)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).astype(np.uint8)
    return packed, sc.astype(np.uint8)
