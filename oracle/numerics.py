"""Exact decoding of stored 16-bit floats and the FP8 E4M3 codec, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

E4M3 here is the "fn" variant used by the pages' FP8 paths (torch.float8_e4m3fn):
1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities, one NaN
code per sign (S.1111.111), largest finite magnitude 448 (S.1111.110), subnormals
m/8 * 2^-6. "Cast" in "Q_fp8 = cast(Q * quant_scale_q)" ("Sparse MLA", RoPE and FP8
quantization) is read as round-to-nearest-even with saturation to +-448 for finite
overflow (and for infinities), NaN kept as NaN.
"""

import numpy as np


def bf16_bits_to_f64(bits):
    """bfloat16 bit patterns (uint16) -> float64, exactly (bf16 is the top half of fp32)."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def fp16_bits_to_f64(bits):
    """IEEE binary16 bit patterns (uint16) -> float64, from the format definition."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    m = (b & 0x3FF).astype(np.float64)
    normal = sign * np.ldexp(1.0 + m / 1024.0, (e - 15).astype(np.int32))
    sub = sign * np.ldexp(m / 1024.0, -14)
    special = np.where(m == 0, sign * np.inf, np.nan)
    return np.where(e == 0, sub, np.where(e == 31, special, normal))


def bits_to_f64(bits, dtype):
    """Decode stored 16-bit values named by ``dtype`` ('bf16' or 'fp16')."""
    if dtype == "bf16":
        return bf16_bits_to_f64(bits)
    if dtype == "fp16":
        return fp16_bits_to_f64(bits)
    raise ValueError(dtype)


E4M3_MAX = 448.0


def e4m3_decode(codes):
    """E4M3 codes (uint8) -> float64."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, np.ldexp(m, -9),
                   np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int32)))
    val = np.where((e == 15) & ((c & 7) == 7), np.nan, val)
    return sign * val


def e4m3_encode(x):
    """float64 -> E4M3 codes: one round-to-nearest-even step, saturating to +-448."""
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    # The spacing of E4M3 values around a: 2^(floor(log2 a) - 3) for normal magnitudes,
    # 2^-9 below the smallest normal 2^-6.
    _, ex = np.frexp(np.where(a == 0, 1.0, a))
    flog = np.maximum(ex - 1, -6)
    with np.errstate(over="ignore", invalid="ignore"):
        quantum = np.ldexp(1.0, (flog - 3).astype(np.int32))
        n = np.rint(np.where(np.isinf(a), 0.0, a) / quantum)  # rint: ties to even
        v = n * quantum
    v = np.where(np.isinf(a), E4M3_MAX, v)
    v = np.minimum(v, E4M3_MAX)
    # Encode the (now representable) magnitude v.
    _, ev = np.frexp(np.where(v == 0, 1.0, v))
    E = ev - 1
    is_sub = (v < 2.0 ** -6)
    field = np.where(is_sub, 0, E + 7)
    mant_sub = np.ldexp(v, 9)
    mant_norm = (np.ldexp(v, (-E).astype(np.int32)) - 1.0) * 8.0
    mant = np.where(is_sub, mant_sub, mant_norm)
    code = (np.where(v == 0, 0, field).astype(np.int64) << 3) | np.where(v == 0, 0, mant).astype(np.int64)
    code = np.where(nan, 0x7F, code)
    code = code | np.where(neg, 0x80, 0)
    return code.astype(np.uint8)


def e4m3_ulp_distance(a, b):
    """|ord(a) - ord(b)| in sign-magnitude order (+0 and -0 both map to 0).

    NaN codes get a distance of 0 when both are NaN and 1000 otherwise.
    """
    a = np.asarray(a, dtype=np.uint8).astype(np.int64)
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)

    def order(c):
        mag = c & 0x7F
        return np.where(c & 0x80, -mag, mag)

    nan_a = (a & 0x7F) == 0x7F
    nan_b = (b & 0x7F) == 0x7F
    d = np.abs(order(a) - order(b))
    d = np.where(nan_a & nan_b, 0, np.where(nan_a | nan_b, 1000, d))
    return d
