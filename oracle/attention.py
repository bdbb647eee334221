"""Exact paged-KV attention in float64 (oracle).

Definition followed (FastDeploy append_attention_c8_impl.cuh,
multi_query_append_attention_c8_kernel and ..._warp1_4_kernel: the block-table
gather, the per-head / per-channel scale registers, the causal bound
``kv_len - q_len + (row token) `` and the chunk bounds; XQA mla_sm120.cu,
kernel_mha: one latent head, V = leading 512 entries of each K row, a single
cache scale for K and V):

For sequence b with q_len = seq_lens[b] query tokens and kvtot = seq_lens_kv[b]
+ q_len cache positions (the appended tokens already sit in the cache at
positions seq_lens_kv[b] .. kvtot-1), query token i (global row
t = cu_seqlens_q[b] + i) and query head h (kv head kvh = h // G):

    position j is visible  iff  j < kvtot  and  (not causal or j <= seq_lens_kv[b] + i)
    page = block_table[b, j // B],  offset = j % B
    k_j[d] = dec(cache_k[page, kvh, offset, d]) * sk(kvh, d)
    v_j[d] = dec(cache_v[page, kvh, d, offset]) * sv(kvh, d)      (V stored transposed)
      (MLA: row = cache[page, offset, :], k_j = row[:Dqk], v_j = row[:Dv], one scale)
    s_j = sm_scale * sum_d q[t, h, d] * k_j[d]          (q is the exact bf16 value)
    lse = log sum_j exp(s_j)                            (natural log, shift by the max)
    out = sum_j exp(s_j - lse) * v_j

A split into KV chunks [lo, hi) gives per-chunk states (m, d, o):
    m = max over visible j in the chunk, d = sum exp(s_j - m), o = sum exp(s_j - m) v_j / d
(m = -inf, d = 0, o = 0 for a chunk with no visible position), and they merge by
    M = max_c m_c,  w_c = d_c exp(m_c - M),  out = sum_c w_c o_c / sum_c w_c,
    lse = M + log sum_c w_c
(FlashInfer persistent.cuh, BlockBatchReductionPersistent / state merge; XQA
mla_sm120.cu, mergePartialOutputs).

Cache access goes through ``page_k(p)`` / ``page_v(p)`` callables that return
one physical page (all kv heads), so multi-GB caches can be regenerated page by
page instead of being held in memory.
"""
from __future__ import annotations

import math
from typing import Callable, Iterable, Optional, Sequence, Tuple

import numpy as np

from .formats import decode_table, bf16_to_f64


def _scales(p, which: str, kvh: int) -> np.ndarray:
    """Scale for kv head kvh: scalar (per head / global) or vector over d (per channel)."""
    s = p.k_scale if which == "k" else p.v_scale
    dim = p.head_dim_qk if which == "k" else p.head_dim_v
    if p.scale_kind == "per_kv_head":
        return bf16_to_f64(np.asarray(s)[kvh:kvh + 1])[0]
    if p.scale_kind == "per_channel":
        return bf16_to_f64(np.asarray(s)[kvh * dim:(kvh + 1) * dim])
    if p.scale_kind == "global":
        return float(np.asarray(s, dtype=np.float32)[0])
    raise ValueError(p.scale_kind)


def _page_accessors(p):
    if hasattr(p, "page_k"):
        return p.page_k, p.page_v
    ck, cv = p.cache_k, p.cache_v
    return (lambda g: ck[g]), (lambda g: cv[g])


def gather_raw(p, b: int, kvh: int, upto: int,
               page_k: Optional[Callable] = None, page_v: Optional[Callable] = None
               ) -> Tuple[np.ndarray, np.ndarray]:
    """Raw cache bytes of positions 0..upto-1 of sequence b, kv head kvh.

    Returns (K [upto, Dqk] uint8, V [upto, Dv] uint8) with V already laid out
    one position per row.
    """
    if page_k is None:
        page_k, page_v = _page_accessors(p)
    B = p.block_size
    nblk = (upto + B - 1) // B
    ks, vs = [], []
    for lb in range(nblk):
        pg = int(p.block_table[b, lb])
        if p.layout == "mla":
            rows = np.asarray(page_k(pg))            # [B, Dqk]
            ks.append(rows)
            vs.append(rows[:, :p.head_dim_v])
        else:
            ks.append(np.asarray(page_k(pg))[kvh])   # [B, D]
            vs.append(np.asarray(page_v(pg))[kvh].T)  # [D, B] -> [B, D]
    if not ks:
        return (np.zeros((0, p.head_dim_qk), np.uint8), np.zeros((0, p.head_dim_v), np.uint8))
    K = np.concatenate(ks, axis=0)[:upto]
    V = np.concatenate(vs, axis=0)[:upto]
    return K, V


def dequant_kv(p, b: int, kvh: int, upto: int, page_k=None, page_v=None):
    """Dequantised K [upto, Dqk] and V [upto, Dv] in float64."""
    Kr, Vr = gather_raw(p, b, kvh, upto, page_k, page_v)
    tab = decode_table(p.kv_dtype)
    K = tab[Kr] * _scales(p, "k", kvh)
    V = tab[Vr] * _scales(p, "v", kvh)
    return K, V


def q_rows(p, b: int, kvh: int) -> np.ndarray:
    """bf16 query values [q_len, G, Dqk] (float64) of sequence b for kv head kvh's group."""
    G = p.q_heads // p.kv_heads
    t0, t1 = int(p.cu_seqlens_q[b]), int(p.cu_seqlens_q[b + 1])
    D = p.head_dim_qk
    bits = np.asarray(p.q_bits)[t0:t1, kvh * G * D:(kvh + 1) * G * D]
    return bf16_to_f64(bits).reshape(t1 - t0, G, D)


def _visible(p, b: int, q_len: int, kvtot: int, lo: int, hi: int) -> np.ndarray:
    """Boolean [q_len, kvtot] mask: causal bound, sequence end and chunk [lo, hi).

    With a speculative tree mask (FastDeploy append_attention_c8_impl.cuh,
    attn_mask [bsz, max_q, max_q] among the draft tokens), appended position
    seq_lens_kv + c is visible to appended token i only if attn_mask[b, i, c]
    is set; the cached prefix stays visible to every token.
    """
    j = np.arange(kvtot)[None, :]
    i = np.arange(q_len)[:, None]
    vis = (j >= lo) & (j < hi)
    pre = int(p.seq_lens_kv[b])
    if p.causal:
        vis = vis & (j <= pre + i)
    mask = getattr(p, "attn_mask", None)
    if mask is not None:
        c = np.clip(j - pre, 0, mask.shape[2] - 1)
        tm = np.asarray(mask[b])[np.arange(q_len)[:, None], c] != 0
        vis = vis & ((j < pre) | tm)
    return vis


def unit_scores(p, b: int, kvh: int, page_k=None, page_v=None):
    """Scores s [q_len, G, kvtot] and dequantised V for one (sequence, kv head)."""
    q_len = int(p.seq_lens[b])
    kvtot = int(p.seq_lens_kv[b]) + q_len
    K, V = dequant_kv(p, b, kvh, kvtot, page_k, page_v)
    Q = q_rows(p, b, kvh)                                   # [q_len, G, D]
    S = p.sm_scale * np.einsum("igd,jd->igj", Q, K)
    return S, V, kvtot


def unit_attention(p, b: int, kvh: int, page_k=None, page_v=None):
    """Full attention for one (sequence, kv head): out [q_len, G, Dv], lse [q_len, G]."""
    S, V, kvtot = unit_scores(p, b, kvh, page_k, page_v)
    q_len = S.shape[0]
    vis = _visible(p, b, q_len, kvtot, 0, kvtot)[:, None, :]
    Sm = np.where(vis, S, -np.inf)
    m = Sm.max(axis=2, keepdims=True) if kvtot > 0 else np.full(S.shape[:2] + (1,), -np.inf)
    safe_m = np.where(np.isfinite(m), m, 0.0)
    e = np.where(vis, np.exp(Sm - safe_m), 0.0)
    z = e.sum(axis=2, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(z > 0, safe_m + np.log(z), -np.inf)
        w = np.where(z > 0, e / np.where(z > 0, z, 1.0), 0.0)
    out = np.einsum("igj,jd->igd", w, V)
    return out, lse[:, :, 0]


def unit_partials(p, b: int, kvh: int, bounds: Sequence[Tuple[int, int]],
                  page_k=None, page_v=None):
    """Per-chunk states for one (sequence, kv head).

    bounds: list of [lo, hi) position ranges.  Returns m, d [C, q_len, G] and
    o [C, q_len, G, Dv] with the conventions of the module docstring.
    """
    S, V, kvtot = unit_scores(p, b, kvh, page_k, page_v)
    q_len, G = S.shape[:2]
    C = len(bounds)
    M = np.full((C, q_len, G), -np.inf)
    Dn = np.zeros((C, q_len, G))
    O = np.zeros((C, q_len, G, V.shape[1]))
    for c, (lo, hi) in enumerate(bounds):
        vis = _visible(p, b, q_len, kvtot, lo, hi)[:, None, :]
        if not vis.any():
            continue
        Sm = np.where(vis, S, -np.inf)
        m = Sm.max(axis=2)
        safe = np.where(np.isfinite(m), m, 0.0)
        e = np.where(vis, np.exp(Sm - safe[:, :, None]), 0.0)
        d = e.sum(axis=2)
        M[c] = m
        Dn[c] = d
        with np.errstate(divide="ignore", invalid="ignore"):
            O[c] = np.where(d[:, :, None] > 0,
                            np.einsum("igj,jd->igd", e, V) / np.where(d > 0, d, 1.0)[:, :, None],
                            0.0)
    return M, Dn, O


def merge_states(M: np.ndarray, Dn: np.ndarray, O: np.ndarray):
    """Log-sum-exp merge over axis 0 of chunk states -> (out, lse)."""
    Mx = M.max(axis=0)
    finite = np.isfinite(Mx)
    safe = np.where(finite, Mx, 0.0)
    with np.errstate(invalid="ignore"):
        w = np.where(np.isfinite(M), Dn * np.exp(np.where(np.isfinite(M), M, 0.0) - safe[None]), 0.0)
    W = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        out = np.where((W > 0)[..., None],
                       np.einsum("c...,c...d->...d", w, O) / np.where(W > 0, W, 1.0)[..., None], 0.0)
        lse = np.where(W > 0, safe + np.log(np.where(W > 0, W, 1.0)), -np.inf)
    return out, lse


def reference(p, units: Optional[Iterable[Tuple[int, int]]] = None, page_k=None, page_v=None):
    """Attention output for the whole problem (or only the listed (b, kvh) units).

    Returns out [T, Hq, Dv] and lse [T, Hq] in float64; rows of units not
    computed are NaN.
    """
    T = int(p.cu_seqlens_q[-1])
    G = p.q_heads // p.kv_heads
    out = np.full((T, p.q_heads, p.head_dim_v), np.nan)
    lse = np.full((T, p.q_heads), np.nan)
    if units is None:
        units = [(b, h) for b in range(len(p.seq_lens)) for h in range(p.kv_heads)]
    for b, kvh in units:
        if int(p.seq_lens[b]) == 0:
            continue
        o, l = unit_attention(p, b, kvh, page_k, page_v)
        t0 = int(p.cu_seqlens_q[b])
        out[t0:t0 + o.shape[0], kvh * G:(kvh + 1) * G] = o
        lse[t0:t0 + o.shape[0], kvh * G:(kvh + 1) * G] = l
    return out, lse


def reference_split(p, chunk: int, units=None, page_k=None, page_v=None):
    """Same result through fixed-size chunks [c*chunk, (c+1)*chunk) plus the merge."""
    T = int(p.cu_seqlens_q[-1])
    G = p.q_heads // p.kv_heads
    out = np.full((T, p.q_heads, p.head_dim_v), np.nan)
    lse = np.full((T, p.q_heads), np.nan)
    if units is None:
        units = [(b, h) for b in range(len(p.seq_lens)) for h in range(p.kv_heads)]
    for b, kvh in units:
        q_len = int(p.seq_lens[b])
        if q_len == 0:
            continue
        kvtot = int(p.seq_lens_kv[b]) + q_len
        n = max(1, math.ceil(kvtot / chunk))
        bounds = [(c * chunk, min(kvtot, (c + 1) * chunk)) for c in range(n)]
        M, Dn, O = unit_partials(p, b, kvh, bounds, page_k, page_v)
        o, l = merge_states(M, Dn, O)
        t0 = int(p.cu_seqlens_q[b])
        out[t0:t0 + q_len, kvh * G:(kvh + 1) * G] = o
        lse[t0:t0 + q_len, kvh * G:(kvh + 1) * G] = l
    return out, lse
