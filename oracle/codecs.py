"""Number formats used by the fp8_ds_mla cache and the MXFP8 output (oracle side).

Everything here follows the format definitions, not any kernel:

* FP8 E4M3 ("e4m3fn", OCP 8-bit floating point): 1 sign bit, 4 exponent bits with
  bias 7, 3 mantissa bits; exponent field 0 is subnormal (value m/8 * 2^-6); there is
  no infinity; S.1111.111 is NaN; the largest finite magnitude is 1.75 * 2^8 = 448.
* bfloat16: the upper 16 bits of an IEEE binary32.
* UE8M0 (OCP MX scale): an unsigned 8-bit biased exponent, value 2^(code - 127),
  code 255 is NaN.
* MX block scale rule (OCP MX, applied to FP8 E4M3 elements): for a block with
  largest magnitude ``amax``, the shared exponent is floor(log2(amax)) - emax_elem,
  with emax_elem = 8 for E4M3; elements are divided by 2^shared_exp and converted
  with round-to-nearest-even, saturating to +-448.

The page that defines the MXFP8 epilogue ("[DSV4.1] Combine DSpark decode and
prefill kernel optimizations", SGLang PR #39370, first description block) states that
the epilogue uses the same UE8M0 conversion as the stock MXFP8 quantizer; the OCP rule
above is the reading taken here (there is no further detail on the pages).
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_EMAX = 8           # exponent of the largest normal (448 = 1.75 * 2^8)
E4M3_MIN_NORMAL_EXP = -6
E4M3_SUBNORMAL_STEP_EXP = -9   # subnormal spacing 2^-9
E4M3_NAN_CODE = 0x7F


def e4m3_decode(codes) -> np.ndarray:
    """Decode E4M3 codes (uint8 array) to float64 values, NaN for S.1111.111.

    Format: OCP FP8 E4M3, the element format of the fp8_ds_mla cache and of the MXFP8 output.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = (c >> 7) & 1
    exp_field = (c >> 3) & 0xF
    mant = c & 0x7
    normal = np.ldexp(1.0 + mant / 8.0, (exp_field - 7).astype(np.int64))
    subnormal = np.ldexp(mant / 8.0, E4M3_MIN_NORMAL_EXP)
    mag = np.where(exp_field == 0, subnormal, normal)
    mag = np.where((exp_field == 0xF) & (mant == 0x7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def _floor_log2(a: np.ndarray) -> np.ndarray:
    """floor(log2(a)) for positive finite float64 a, exactly (via frexp)."""
    _, e = np.frexp(a)          # a = f * 2^e, f in [0.5, 1)
    return e.astype(np.int64) - 1


def e4m3_encode(x) -> np.ndarray:
    """Round float64 values to E4M3 codes: round-to-nearest-even, saturate to +-448.

    NaN maps to the NaN code 0x7F.  The sign of zero is kept (0x80 for -0 and for
    negative values that round to zero).

    Format: OCP FP8 E4M3 with round-to-nearest-even and saturation (a reading).
    """
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    a = np.minimum(a, 1e300)                     # keep +inf finite for the arithmetic below
    pos = a > 0
    e = np.where(pos, _floor_log2(np.where(pos, a, 1.0)), E4M3_MIN_NORMAL_EXP)
    e = np.maximum(e, E4M3_MIN_NORMAL_EXP)       # below 2^-6 the spacing is fixed at 2^-9
    step_exp = e - 3                             # 3 mantissa bits
    q = np.round(np.ldexp(a, -step_exp)) * 1.0   # np.round: ties to even
    mag = np.ldexp(q, step_exp)
    mag = np.minimum(mag, E4M3_MAX)              # satfinite
    # encode the (now representable) magnitude
    is_normal = mag >= np.ldexp(1.0, E4M3_MIN_NORMAL_EXP)
    me = np.where(is_normal, _floor_log2(np.where(is_normal, mag, 1.0)), 0)
    mant_normal = np.round((np.ldexp(mag, -me) - 1.0) * 8.0).astype(np.int64)
    field_normal = (me + 7).astype(np.int64)
    mant_sub = np.round(np.ldexp(mag, -E4M3_SUBNORMAL_STEP_EXP)).astype(np.int64)
    code = np.where(is_normal, (field_normal << 3) | mant_normal, mant_sub)
    code = np.where(neg, code | 0x80, code)
    code = np.where(nan, E4M3_NAN_CODE, code)
    return code.astype(np.uint8)


def e4m3_ulp_distance(a_codes, b_codes) -> np.ndarray:
    """Distance between two E4M3 codes counted in steps of the E4M3 value lattice.

    Both codes must be finite.  Positive and negative zero are the same point.

    Used by the FP8-code matching criterion of the tests, not by the path itself.
    """
    def ordinal(c):
        c = np.asarray(c, dtype=np.uint8).astype(np.int64)
        mag = c & 0x7F
        return np.where((c & 0x80) != 0, -mag, mag)
    return np.abs(ordinal(a_codes) - ordinal(b_codes))


def bf16_decode(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) to float64.

    Format: bfloat16, the type of q, the norm weight and the rope part of a cache row.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def bf16_encode(x) -> np.ndarray:
    """Round float64 values to bfloat16 bit patterns (uint16): round-to-nearest-even on
    the binary32 value's upper half.  x is first rounded to binary32 (the values this
    oracle rounds are binary32 or exact in it); NaN gives the quiet NaN 0x7FC0, +-inf stay
    infinite.

    Format: bfloat16, the rope part of a cache row written by the KV insert.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint32)
    r = np.where(np.isnan(f), 0x7FC0, r)
    return r.astype(np.uint16)


def fp32_decode_le(raw) -> np.ndarray:
    """Little-endian IEEE binary32 from a uint8 array whose last axis is a multiple of 4.

    Format: IEEE binary32, the per-128 scales of an fp8_ds_mla row.
    """
    r = np.ascontiguousarray(np.asarray(raw, dtype=np.uint8))
    return r.view("<f4").astype(np.float64)


def ue8m0_decode(codes) -> np.ndarray:
    """UE8M0 codes to their scale 2^(code - 127), NaN for code 255.

    Format: OCP MX scale (a reading)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    v = np.ldexp(1.0, c - 127)
    return np.where(c == 255, np.nan, v)


def mx_shared_exponent(amax) -> np.ndarray:
    """Shared exponent of an MX block with E4M3 elements: floor(log2 amax) - 8,
    clamped to the UE8M0 range [-127, 127]; a block of zeros takes -127 (code 0).

    Rule: OCP MX for E4M3 elements, the UE8M0 conversion that "[DSV4.1] Combine DSpark
    decode and prefill kernel optimizations" (SGLang PR #39370), first description block
    refers to (a reading).
    """
    a = np.asarray(amax, dtype=np.float64)
    pos = a > 0
    e = np.where(pos, _floor_log2(np.where(pos, a, 1.0)) - E4M3_EMAX, -127)
    return np.clip(e, -127, 127).astype(np.int64)


def mxfp8_quantize(x, block: int = 32):
    """MXFP8 cast along the last axis: returns (E4M3 codes, UE8M0 scale codes).

    The last axis must be a multiple of ``block``.  Each block's elements are divided
    by 2^E (E = ``mx_shared_exponent`` of the block's largest magnitude) and rounded
    to E4M3 with ties to even and saturation.

    Rule: OCP MX block quantisation, the MXFP8 epilogue of "[DSV4.1] Combine DSpark decode
    and prefill kernel optimizations" (SGLang PR #39370), first description block (a
    reading).
    """
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    assert n % block == 0
    xb = x.reshape(x.shape[:-1] + (n // block, block))
    amax = np.max(np.abs(xb), axis=-1)
    e = mx_shared_exponent(amax)
    scaled = np.ldexp(xb, -e[..., None])
    codes = e4m3_encode(scaled).reshape(x.shape)
    sf = (e + 127).astype(np.uint8)
    return codes, sf


def sf_swizzle_128x4(sf) -> np.ndarray:
    """Scale codes [M, K] (K a multiple of 4) laid out in 128 x 4 tiles, as the bytes of
    FlashInfer's 128x4 scale-factor swizzle; rows M..ceil(M/128)*128 - 1 are zero.

    The page ("[DSV4.1] Combine DSpark decode and prefill kernel optimizations", SGLang
    PR #39370, mHC MXFP8 epilogue paragraph) names the layout but prints no byte order;
    the reading taken: tiles of 128 rows x 4 columns, 512 bytes each, in row-major tile
    order; inside a tile, row m and column k sit at (m % 32) * 16 + (m // 32) * 4 + k,
    so that the four 32-row quarters of the tile interleave at a 4-byte stride and a
    row's four codes are adjacent.  Written out entry by entry from that description.
    """
    sf = np.asarray(sf, dtype=np.uint8)
    M, K = sf.shape
    assert K % 4 == 0
    m_pad = -(-M // 128) * 128
    out = np.zeros(m_pad * K, dtype=np.uint8)
    tiles_per_row = K // 4
    for m in range(M):
        for k in range(K):
            tile = (m // 128) * tiles_per_row + k // 4
            r, c = m % 128, k % 4
            out[tile * 512 + (r % 32) * 16 + (r // 32) * 4 + c] = sf[m, k]
    return out
