"""Bit-level decoders for the cache and query element types (oracle; test only).

The pages fix the cache element type only by name: an FP8 latent KV cache with a
single per-tensor scale ("Context Parallel Guide (PCP & DCP)", DCP Guide, Tips
and "How it works" item 4: "fp8 KV cache. Per-tensor scale"; per-token and
per-group layouts are not supported). The format itself is the OCP 8-bit
floating point E4M3 ("fn") encoding, which this module writes out from its
definition:

* 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
* exponent field 0 encodes subnormals ``(-1)^s * (m/8) * 2^-6``;
* there is no infinity; the two codes with all exponent and mantissa bits set
  (0x7F and 0xFF) are NaN; every other code is finite, the largest 448.

BF16 is the upper half of an IEEE-754 binary32 word.
"""

from __future__ import annotations

import math

import numpy as np


def e4m3_value(code: int) -> float:
    """Value of one E4M3 code, from the OCP definition (NaN for 0x7F/0xFF)."""
    code = int(code) & 0xFF
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp_field = (code >> 3) & 0xF
    mant = code & 0x7
    if exp_field == 0xF and mant == 0x7:
        return math.nan
    if exp_field == 0:
        return sign * (mant / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)


#: float64 value of each of the 256 E4M3 codes.
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """Decode an array of uint8 E4M3 codes to float64 (exact)."""
    codes = np.asarray(codes)
    if codes.dtype != np.uint8:
        raise TypeError("E4M3 codes must be uint8")
    return E4M3_TABLE[codes]


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """Decode an array of uint16 BF16 bit patterns to float64 (exact)."""
    bits = np.asarray(bits)
    if bits.dtype != np.uint16:
        raise TypeError("BF16 bit patterns must be uint16")
    words = bits.astype(np.uint32) << np.uint32(16)
    return words.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest BF16 (ties to even), as float64.

    Used only to express the final output's element type when a test forms the
    half-ulp allowance; the comparison itself stays in float64.
    """
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    w = x32.view(np.uint32).astype(np.uint64)
    lsb = (w >> np.uint64(16)) & np.uint64(1)
    w = (w + np.uint64(0x7FFF) + lsb) >> np.uint64(16) << np.uint64(16)
    out = w.astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(x32)
    out[nan] = np.nan
    return out


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of BF16 numbers at |x| (2^(e-7) for |x| in [2^e, 2^(e+1)))."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    tiny = 2.0 ** -133
    e = np.floor(np.log2(np.maximum(ax, tiny)))
    e = np.maximum(e, -126.0)
    return 2.0 ** (e - 7)
