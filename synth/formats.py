"""Storage-format helpers for building synthetic inputs (host side).

These round real numbers into the storage types the workloads use (bf16 for
queries and scales, OCP FP8 E4M3 for fp8 caches).  They only PREPARE inputs;
the quantities the attention path computes are never formed here.  Rounding is
delegated to PyTorch's CPU dtype conversions (round to nearest even).
"""
from __future__ import annotations

import numpy as np
import torch

E4M3_MAX = 448.0


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float array -> bf16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    """float array -> E4M3 codes (uint8), saturated to +-448, round to nearest even."""
    xc = np.clip(np.asarray(x, dtype=np.float32), -E4M3_MAX, E4M3_MAX)
    t = torch.from_numpy(np.ascontiguousarray(xc))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def int8_to_bytes(v: np.ndarray) -> np.ndarray:
    """signed integers in [-128, 127] -> two's-complement bytes (uint8)."""
    return np.asarray(v, dtype=np.int64).astype(np.int8).view(np.uint8)
