"""Quantise-and-write of the appended tokens' K / V into the paged cache (oracle).

Test infrastructure only, like the rest of ``oracle/``.

The attention pages (FastDeploy append_attention_c8_impl.cuh) read the
appended tokens' keys and values from the int8 / FP8 cache: the writer runs
before them and is not on the pages, so this follows the conventions the
attention path reads (same layouts, real = stored x scale):

  token i of sequence b (global row t = cu_seqlens_q[b] + i) goes to cache
  position j = seq_lens_kv[b] + i, page = block_table[b, j // B], offset j % B;
  stored = Q(x / s) for the bf16 input value x and the scale s of its (kv head,
  channel) (per kv head, per channel, or one global fp32 scale):
    - the quotient is the IEEE binary32 division of the two fp32 values (the
      precision in which the kernel takes the decision);
    - int8: round half to even, saturate to [-127, 127], two's-complement byte;
    - E4M3: nearest finite E4M3 value, ties to the even mantissa, |v| > 448
      saturates to +-448, the sign of zero kept.
  GQA: K[page, kvh, offset, d] and V[page, kvh, d, offset] (V transposed per
  page).  MLA: cache[page, offset, :] = Q(the token's latent row), one scale.
"""
from __future__ import annotations

import numpy as np

from .formats import e4m3_value, bf16_to_f64

E4M3_MAX = 448.0

# finite non-negative E4M3 values and their codes (0x00 .. 0x7E)
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = np.array([e4m3_value(int(c)) for c in _POS_CODES], dtype=np.float64)


def e4m3_encode(v) -> np.ndarray:
    """float32 values -> E4M3 codes by direct search over the finite values:
    the nearest one, ties to the even mantissa (code LSB 0), saturation at 448."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    d = np.abs(a[..., None] - _POS_VALUES)                 # distance to every finite value
    best = d.min(axis=-1, keepdims=True)
    cand = d == best                                       # one or two nearest codes
    even = cand & ((_POS_CODES & 1) == 0)
    pick = np.where(even.any(axis=-1, keepdims=True), even, cand)
    code = np.argmax(pick, axis=-1).astype(np.uint8)
    neg = np.signbit(v)
    return np.where(neg, code | np.uint8(0x80), code).astype(np.uint8)


def int8_encode(v) -> np.ndarray:
    """float32 values -> int8 codes: round half to even, saturate to +-127."""
    r = np.rint(np.asarray(v, dtype=np.float32).astype(np.float64))
    return np.clip(r, -127, 127).astype(np.int64).astype(np.int8).view(np.uint8)


def quantize(x_bits, scale, kv_dtype: str) -> np.ndarray:
    """bf16 bit patterns and fp32 scales (broadcast) -> stored bytes."""
    x = bf16_to_f64(x_bits).astype(np.float32)
    q = x / np.asarray(scale, dtype=np.float32)            # binary32 division
    return e4m3_encode(q) if kv_dtype == "fp8_e4m3" else int8_encode(q)


def _scales(p, scale, kvh: int, D: int) -> np.ndarray:
    """fp32 scale of each channel of kv head kvh."""
    if p.scale_kind == "global":
        return np.full(D, np.float32(np.asarray(scale, np.float32).reshape(-1)[0]))
    s = bf16_to_f64(np.asarray(scale, np.uint16)).astype(np.float32)
    if p.scale_kind == "per_kv_head":
        return np.full(D, s[kvh])
    return s[kvh * D:(kvh + 1) * D]


def cache_append(p, k_new_bits, v_new_bits, cache_k, cache_v):
    """Write the appended tokens of problem ``p`` into copies of the caches.

    k_new_bits / v_new_bits: uint16 bf16 bits [T, kv_heads, Dqk] / [T, kv_heads,
    Dv] (MLA: k_new_bits [T, Dqk], v_new_bits unused).  Returns (cache_k,
    cache_v) as new arrays.
    """
    ck = np.array(cache_k, copy=True)
    cv = None if cache_v is None else np.array(cache_v, copy=True)
    B = p.block_size
    for b in range(len(p.seq_lens)):
        for i in range(int(p.seq_lens[b])):
            t = int(p.cu_seqlens_q[b]) + i
            j = int(p.seq_lens_kv[b]) + i
            page = int(p.block_table[b, j // B])
            off = j % B
            if p.layout == "mla":
                s = _scales(p, p.k_scale, 0, p.head_dim_qk)
                ck[page, off, :] = quantize(k_new_bits[t], s, p.kv_dtype)
                continue
            for kvh in range(p.kv_heads):
                sk = _scales(p, p.k_scale, kvh, p.head_dim_qk)
                sv = _scales(p, p.v_scale, kvh, p.head_dim_v)
                ck[page, kvh, off, :] = quantize(k_new_bits[t, kvh], sk, p.kv_dtype)
                cv[page, kvh, :, off] = quantize(v_new_bits[t, kvh], sv, p.kv_dtype)
    return ck, cv
