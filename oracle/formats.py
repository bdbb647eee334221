"""Decoding of the stored element formats (oracle side, fp64).

int8 (FastDeploy append_attention_c8_impl.cuh, CacheT = uint8_t storage with
the IsFP8 = false instantiation): a byte is read as a signed two's-complement
integer; the real value is that integer times the cache scale (no zero point:
the cache_k_zp / cache_v_zp tensors are accepted but never passed on).

FP8 E4M3 (same file with IsFP8 = true; XQA mla_sm120.cu with an E4M3 cache
element and kE4M3_MAX = 448), OCP FP8 definition:
  bit 7 sign, bits 6..3 exponent E (bias 7), bits 2..0 mantissa M;
  E = 0      : (-1)^s * M/8 * 2^(1-7)            (subnormal)
  E = 15,M=7 : NaN                                (no infinities)
  otherwise  : (-1)^s * (1 + M/8) * 2^(E-7)
"""
from __future__ import annotations

import numpy as np


def int8_value(code: int) -> float:
    c = int(code) & 0xFF
    return float(c - 256 if c >= 128 else c)


def e4m3_value(code: int) -> float:
    c = int(code) & 0xFF
    s = -1.0 if (c >> 7) else 1.0
    e = (c >> 3) & 0xF
    m = c & 0x7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** (1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def decode_table(kv_dtype: str) -> np.ndarray:
    """256-entry float64 table: byte code -> stored real value (before scaling)."""
    f = int8_value if kv_dtype == "int8" else e4m3_value
    return np.array([f(c) for c in range(256)], dtype=np.float64)


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64: the top half of an IEEE binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)
