"""NVFP4 decoding for the oracle (float64). TEST INFRASTRUCTURE ONLY.

Muse Spark Open Ultrafast, section "The model": experts are stored in 4-bit
NVFP4. The page gives no format details, so this follows the published NVFP4
layout: e2m1 element codes, one e4m3 scale per block of 16 consecutive elements
along the reduction dimension, and one float32 scale per (expert, projection)
tensor:

    w[r, k] = e2m1(code[r, k]) * e4m3(scale[r, k // 16]) * tensor_scale

Byte layout (a documented choice): codes are packed two per byte along k, the
even k in the low nibble; scales are one byte per block, row-major.
"""

from __future__ import annotations

import numpy as np


def e2m1_value(code: int) -> float:
    """Value of a 4-bit e2m1 code: 1 sign, 2 exponent (bias 1), 1 mantissa bit.

    Exponent field 0 is subnormal: 0.5 * mantissa. Otherwise
    2**(exp - 1) * (1 + mantissa / 2). No infinities or NaNs.
    """
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    exp = (code >> 1) & 0x3
    man = code & 0x1
    if exp == 0:
        mag = 0.5 * man
    else:
        mag = 2.0 ** (exp - 1) * (1.0 + man / 2.0)
    return sign * mag


def e4m3_value(byte: int) -> float:
    """Value of an e4m3 (fn variant) byte: 1 sign, 4 exponent (bias 7), 3 mantissa.

    Exponent field 0 is subnormal: 2**-6 * mantissa / 8. Exponent 15 with mantissa
    7 is NaN; there are no infinities, so 0x7E = 448 is the largest finite value.
    """
    byte = int(byte) & 0xFF
    sign = -1.0 if byte & 0x80 else 1.0
    exp = (byte >> 3) & 0xF
    man = byte & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        mag = 2.0 ** -6 * (man / 8.0)
    else:
        mag = 2.0 ** (exp - 7) * (1.0 + man / 8.0)
    return sign * mag


_E2M1 = np.array([e2m1_value(c) for c in range(16)], np.float64)
_E4M3 = np.array([e4m3_value(b) for b in range(256)], np.float64)


def dequant_nvfp4_rows(codes: np.ndarray, scales: np.ndarray, tensor_scale: float) -> np.ndarray:
    """Dequantise rows of NVFP4 weights to float64.

    codes  uint8 [R, K/2]  (element 2i in the low nibble of byte i, 2i+1 in the high)
    scales uint8 [R, K/16] (e4m3 bit patterns, one per 16-element block)
    tensor_scale float     (float32 per-tensor scale)
    Returns float64 [R, K].
    """
    codes = np.asarray(codes, np.uint8)
    scales = np.asarray(scales, np.uint8)
    rows, half = codes.shape
    k = 2 * half
    assert scales.shape == (rows, k // 16)
    out = np.empty((rows, k), np.float64)
    out[:, 0::2] = _E2M1[codes & 0xF]
    out[:, 1::2] = _E2M1[codes >> 4]
    block = np.repeat(_E4M3[scales], 16, axis=1)
    return out * block * float(tensor_scale)


def dequant_fp8_block(codes: np.ndarray, scales: np.ndarray, block: int = 128) -> np.ndarray:
    """Dequantise FP8 block-scaled weights to float64.

    codes  uint8 [R, K]  e4m3 bit patterns, one per element
    scales float32 [R / block, K / block], one per block x block tile
    Returns float64 [R, K] = e4m3(code) * scale of the element's tile. (Ling-3.0-flash
    blog, "Where the time goes now": fp8 weights with 128-wide blocks.)
    """
    codes = np.asarray(codes, np.uint8)
    scales = np.asarray(scales, np.float64)
    r, k = codes.shape
    assert scales.shape == (r // block, k // block)
    return _E4M3[codes] * np.repeat(np.repeat(scales, block, axis=0), block, axis=1)
