"""Seeded synthetic workloads for paged, quantised-KV attention.

A ``Case`` holds one problem: shapes, per-sequence lengths, the block table,
bf16 queries, scales and the paged int8 / FP8-E4M3 caches.  Every array is a
pure function of (seed, stream, flat index) through ``synth.rng``, so a single
page can be regenerated on the host for a spot check while the full cache is
produced on the device by ``synth/csrc/synth_gen.cu`` (uniform int8 caches).

The five named workloads follow the serving scenarios of the source pages
(FastDeploy append_attention_c8_impl.cuh: decode / speculative verify / chunked
prefill over a block-table int8 or fp8 cache; XQA mla_sm120.cu: MLA decode with
a 576/512 latent head).  Readings where the workload text is silent:
  * fp8 per-kv-head scale = bf16(amax over that head's N(0,1) draws / 448);
  * int8 per-kv-head scale for spec-verify: uniform[0.005, 0.02] like decode;
  * MLA global scale = float32(amax over the whole latent cache / 448);
  * the decode-2 block table takes whole pages from a Fisher-Yates shuffle of
    the 4096-page pool, sequence after sequence; unused entries are -1;
  * the decode-1 block table is an 8-page permutation reshaped to [2, 4].

Layouts (row-major):
  GQA: cache_k [P, Hkv, B, D], cache_v [P, Hkv, D, B]  (V transposed per page)
  MLA: cache   [P, B, Dqk]; V is the first Dv entries of each row.
  q [T, q_stride] bf16 bits, head h of token t at q[t, h*Dqk : (h+1)*Dqk].
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

from . import rng
from .formats import to_bf16_bits, bf16_bits_to_f64, to_e4m3_bytes, int8_to_bytes, E4M3_MAX

# counter streams
S_LEN_KV = 1
S_LEN_Q = 2
S_Q = 3
S_K = 4
S_V = 5
S_KSCALE = 6
S_VSCALE = 7
S_PERM = 8
S_KNEW = 9
S_VNEW = 10
S_TREE = 11

INT8 = "int8"
FP8 = "fp8_e4m3"
PER_HEAD = "per_kv_head"
PER_CHANNEL = "per_channel"
GLOBAL = "global"
GQA = "gqa"
MLA = "mla"

_CHUNK_ELEMS = 1 << 24


@dataclasses.dataclass
class Case:
    name: str
    seed: int
    bsz: int
    q_heads: int
    kv_heads: int
    head_dim_qk: int
    head_dim_v: int
    block_size: int
    num_pages: int
    max_blocks_per_seq: int
    kv_dtype: str
    scale_kind: str
    layout: str
    causal: bool
    chunk_size: int
    sm_scale: float
    q_stride: int
    seq_lens: np.ndarray        # int32 [bsz]  query tokens per sequence
    seq_lens_kv: np.ndarray     # int32 [bsz]  cached prefix length
    cu_seqlens_q: np.ndarray    # int32 [bsz+1]
    block_table: np.ndarray     # int32 [bsz, max_blocks_per_seq]
    q_bits: np.ndarray          # uint16 [T, q_stride] (bf16)
    k_scale: np.ndarray         # uint16 bf16 bits [Hkv] / [Hkv*D], or float32 [1]
    v_scale: np.ndarray
    int8_range: tuple = (-127, 127)
    # optional speculative tree mask [bsz, max_q, max_q] uint8: appended token i
    # of a sequence sees appended token j iff attn_mask[b, i, j] (and j <= i)
    attn_mask: Optional[np.ndarray] = None
    _cache_k: Optional[np.ndarray] = None
    _cache_v: Optional[np.ndarray] = None
    _page_memo: Optional[dict] = None

    # ----- derived sizes -------------------------------------------------
    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def kvtot(self) -> np.ndarray:
        return (self.seq_lens_kv.astype(np.int64) + self.seq_lens.astype(np.int64))

    @property
    def k_shape(self):
        if self.layout == MLA:
            return (self.num_pages, self.block_size, self.head_dim_qk)
        return (self.num_pages, self.kv_heads, self.block_size, self.head_dim_qk)

    @property
    def v_shape(self):
        if self.layout == MLA:
            return self.k_shape
        return (self.num_pages, self.kv_heads, self.head_dim_v, self.block_size)

    @property
    def device_generable(self) -> bool:
        """True when the caches are uniform int8 draws the device generator reproduces."""
        return self.kv_dtype == INT8

    # ----- cache bytes ---------------------------------------------------
    def kv_bytes(self, which: str, start: int, count: int) -> np.ndarray:
        """Bytes [start, start+count) of the flat K ('k') or V ('v') pool."""
        if self.layout == MLA and which == "v":
            which = "k"
        stream = S_K if which == "k" else S_V
        held = self._cache_k if which == "k" else self._cache_v
        if held is not None:
            return held.reshape(-1)[start:start + count]
        if self.kv_dtype == INT8:
            lo, hi = self.int8_range
            return rng.uniform_i8_bytes(self.seed, stream, start, count, lo, hi)
        full = self.cache_k if which == "k" else self.cache_v
        return full.reshape(-1)[start:start + count]

    def _gen_int8(self, which: str) -> np.ndarray:
        shape = self.k_shape if which == "k" else self.v_shape
        n = int(np.prod(shape))
        out = np.empty(n, dtype=np.uint8)
        for s in range(0, n, _CHUNK_ELEMS):
            c = min(_CHUNK_ELEMS, n - s)
            out[s:s + c] = self.kv_bytes(which, s, c)
        return out.reshape(shape)

    @property
    def cache_k(self) -> np.ndarray:
        if self._cache_k is None:
            self._cache_k = self._gen_int8("k")
        return self._cache_k

    @property
    def cache_v(self) -> np.ndarray:
        if self.layout == MLA:
            return self.cache_k
        if self._cache_v is None:
            self._cache_v = self._gen_int8("v")
        return self._cache_v

    def page_k(self, page: int) -> np.ndarray:
        """One physical page of K (all kv heads), regenerated without the rest."""
        return self._page("k", page)

    def page_v(self, page: int) -> np.ndarray:
        return self._page("v", page)

    def _page(self, which: str, page: int) -> np.ndarray:
        if self._page_memo is None:
            self._page_memo = {}
        key = (which, int(page))
        got = self._page_memo.get(key)
        if got is None:
            shape = (self.k_shape if which == "k" else self.v_shape)[1:]
            n = int(np.prod(shape))
            got = self.kv_bytes(which, int(page) * n, n).reshape(shape)
            if len(self._page_memo) < 200_000:
                self._page_memo[key] = got
        return got

    def kv_bytes_total(self) -> int:
        """Cache bytes the attention must read once: every visible (page, head) slab."""
        pages = np.ceil(self.kvtot / self.block_size).astype(np.int64)
        if self.layout == MLA:
            return int(pages.sum()) * self.block_size * self.head_dim_qk
        per = self.block_size * (self.head_dim_qk + self.head_dim_v) * self.kv_heads
        return int(pages.sum()) * per


# ---------------------------------------------------------------------------
def _bf16_uniform(seed, stream, n, a, b):
    return to_bf16_bits(rng.uniform_real(seed, stream, np.arange(n, dtype=np.uint64), a, b))


def _fp8_pool_gqa(seed, stream, shape, kv_heads):
    """fp8 GQA cache from N(0,1) with per-kv-head bf16 scale amax/448."""
    P = shape[0]
    per_page = int(np.prod(shape[1:]))
    per_head = per_page // kv_heads
    # pass 1: amax per head
    amax = np.zeros(kv_heads)
    pages_per_chunk = max(1, _CHUNK_ELEMS // per_page)
    for p0 in range(0, P, pages_per_chunk):
        p1 = min(P, p0 + pages_per_chunk)
        idx = np.arange(p0 * per_page, p1 * per_page, dtype=np.uint64)
        x = rng.normal(seed, stream, idx).reshape(p1 - p0, kv_heads, per_head)
        amax = np.maximum(amax, np.abs(x).max(axis=(0, 2)))
    sbits = to_bf16_bits(amax / E4M3_MAX)
    s = (sbits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    out = np.empty(P * per_page, dtype=np.uint8)
    for p0 in range(0, P, pages_per_chunk):
        p1 = min(P, p0 + pages_per_chunk)
        idx = np.arange(p0 * per_page, p1 * per_page, dtype=np.uint64)
        x = rng.normal(seed, stream, idx).reshape(p1 - p0, kv_heads, per_head)
        out[p0 * per_page:p1 * per_page] = to_e4m3_bytes(x / s[None, :, None]).reshape(-1)
    return out.reshape(shape), sbits


def _fp8_pool_global(seed, stream, shape):
    n = int(np.prod(shape))
    amax = 0.0
    for s0 in range(0, n, _CHUNK_ELEMS):
        c = min(_CHUNK_ELEMS, n - s0)
        amax = max(amax, float(np.abs(rng.normal(seed, stream, np.arange(s0, s0 + c, dtype=np.uint64))).max()))
    scale = np.array([amax / E4M3_MAX], dtype=np.float32)
    out = np.empty(n, dtype=np.uint8)
    for s0 in range(0, n, _CHUNK_ELEMS):
        c = min(_CHUNK_ELEMS, n - s0)
        x = rng.normal(seed, stream, np.arange(s0, s0 + c, dtype=np.uint64))
        out[s0:s0 + c] = to_e4m3_bytes(x / float(scale[0]))
    return out.reshape(shape), scale


def make_case(*, name="custom", seed=1, seq_lens, seq_lens_kv, q_heads, kv_heads,
              head_dim_qk=128, head_dim_v=None, block_size=64, kv_dtype=INT8,
              scale_kind=PER_HEAD, layout=GQA, causal=True, chunk_size=0,
              sm_scale=None, q_stride=None, num_pages=None, extra_blocks=0,
              table="shuffle", int8_range=(-127, 127), scale_range=(0.005, 0.02)):
    """Build a seeded case from explicit per-sequence lengths.

    table: "shuffle" takes each sequence's pages from a Fisher-Yates shuffle of
    the pool; "reshape" fills the whole [bsz, max_blocks] table with the shuffle
    (the decode-1 reading); unused entries are -1 with "shuffle".
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    seq_lens_kv = np.asarray(seq_lens_kv, dtype=np.int32)
    bsz = len(seq_lens)
    if head_dim_v is None:
        head_dim_v = head_dim_qk
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim_qk)
    if q_stride is None:
        q_stride = q_heads * head_dim_qk
    kvtot = seq_lens_kv.astype(np.int64) + seq_lens.astype(np.int64)
    pages_needed = (kvtot + block_size - 1) // block_size
    max_blocks = int(max(1, pages_needed.max() if bsz else 1)) + extra_blocks
    if table == "reshape" and num_pages is not None:
        max_blocks = num_pages // bsz
    if num_pages is None:
        num_pages = int(pages_needed.sum()) if table == "shuffle" else bsz * max_blocks
    perm = rng.permutation(seed, S_PERM, num_pages)
    block_table = np.full((bsz, max_blocks), -1, dtype=np.int32)
    if table == "reshape":
        assert num_pages == bsz * max_blocks
        block_table[:] = perm.reshape(bsz, max_blocks)
    else:
        off = 0
        for b in range(bsz):
            n = int(pages_needed[b])
            assert off + n <= num_pages, "page pool too small for the drawn lengths"
            block_table[b, :n] = perm[off:off + n]
            off += n
    cu = np.zeros(bsz + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seq_lens)
    T = int(cu[-1])
    qv = np.zeros((T, q_stride), dtype=np.float64)
    dense = q_heads * head_dim_qk
    idx = np.arange(T * dense, dtype=np.uint64)
    qv[:, :dense] = rng.normal(seed, S_Q, idx).reshape(T, dense)
    q_bits = to_bf16_bits(qv)

    case = Case(name=name, seed=seed, bsz=bsz, q_heads=q_heads, kv_heads=kv_heads,
                head_dim_qk=head_dim_qk, head_dim_v=head_dim_v, block_size=block_size,
                num_pages=num_pages, max_blocks_per_seq=max_blocks, kv_dtype=kv_dtype,
                scale_kind=scale_kind, layout=layout, causal=bool(causal),
                chunk_size=chunk_size, sm_scale=float(sm_scale), q_stride=q_stride,
                seq_lens=seq_lens, seq_lens_kv=seq_lens_kv, cu_seqlens_q=cu,
                block_table=block_table, q_bits=q_bits, k_scale=None, v_scale=None,
                int8_range=tuple(int8_range))

    if kv_dtype == INT8:
        a, b_ = scale_range
        if scale_kind == PER_HEAD:
            case.k_scale = _bf16_uniform(seed, S_KSCALE, kv_heads, a, b_)
            case.v_scale = _bf16_uniform(seed, S_VSCALE, kv_heads, a, b_)
        elif scale_kind == PER_CHANNEL:
            case.k_scale = _bf16_uniform(seed, S_KSCALE, kv_heads * head_dim_qk, a, b_)
            case.v_scale = _bf16_uniform(seed, S_VSCALE, kv_heads * head_dim_v, a, b_)
        elif scale_kind == GLOBAL:
            s = rng.uniform_real(seed, S_KSCALE, np.arange(1, dtype=np.uint64), a, b_)
            case.k_scale = s.astype(np.float32)
            case.v_scale = case.k_scale.copy()
        else:
            raise ValueError(scale_kind)
    elif kv_dtype == FP8:
        if scale_kind == PER_HEAD:
            assert layout == GQA
            case._cache_k, case.k_scale = _fp8_pool_gqa(seed, S_K, case.k_shape, kv_heads)
            case._cache_v, case.v_scale = _fp8_pool_gqa(seed, S_V, case.v_shape, kv_heads)
        elif scale_kind == GLOBAL:
            case._cache_k, case.k_scale = _fp8_pool_global(seed, S_K, case.k_shape)
            if layout == MLA:
                case.v_scale = case.k_scale.copy()
            else:
                case._cache_v, _ = _fp8_pool_global(seed, S_V, case.v_shape)
                case.v_scale = case.k_scale.copy()
        else:
            raise ValueError("fp8 caches use per-kv-head or global scales")
    else:
        raise ValueError(kv_dtype)
    return case


def _draw_lens(seed, stream, n, lo, hi):
    return rng.uniform_int(seed, stream, np.arange(n, dtype=np.uint64), lo, hi).astype(np.int32)


# The five workloads.  Seed = workload number.
CONFIG_NAMES = {
    1: "decode-1: bsz 2, q_len 1, Hq 4/Hkv 1, D 128, int8 per-head, prefix [100,37], no split",
    2: "decode-2: bsz 64, q_len 1, Hq 32/Hkv 8, D 128, int8 per-channel, prefix U[512,4096], "
       "4096-page pool, chunk 512 + merge",
    3: "append-3: bsz 8, q_len U[64,512], prefix U[0,8192], Hq 32/Hkv 8, D 128, causal, "
       "fp8 per-head, no split",
    4: "spec-verify-4: bsz 128, q_len 6 causal, Hq 64/Hkv 8, D 128, prefix U[8192,32768], "
       "int8 per-head, chunk 1024 + merge",
    5: "mla-5: bsz 32, q_len U{1,2}, 128 q heads / 1 latent, K 576 / V 512, fp8 global scale, "
       "prefix U[4096,16384], scale 1/sqrt(192), split + merge",
}


def config(n: int, bsz_limit: int = 0) -> Case:
    """Workload n; bsz_limit > 0 keeps only its first bsz_limit sequences (the
    same draws), for profiling captures of workloads too large to capture."""
    case = _config(n)
    if bsz_limit <= 0 or bsz_limit >= case.bsz:
        return case
    if n not in (2, 4, 5):
        raise ValueError("bsz_limit applies to the decode-family and MLA workloads")
    return _config(n, bsz_limit)


def _config(n: int, bsz_limit: int = 0) -> Case:
    def cut(name, lens_q, lens_kv):
        if not bsz_limit:
            return name, lens_q, lens_kv
        return f"{name} (first {bsz_limit} sequences)", lens_q[:bsz_limit], lens_kv[:bsz_limit]
    if n == 1:
        return make_case(name="decode-1", seed=1, seq_lens=[1, 1], seq_lens_kv=[100, 37],
                         q_heads=4, kv_heads=1, kv_dtype=INT8, scale_kind=PER_HEAD,
                         causal=True, chunk_size=0, num_pages=8, table="reshape")
    if n == 2:
        bsz = 64
        name, ql, kv = cut("decode-2", np.ones(bsz, np.int32), _draw_lens(2, S_LEN_KV, bsz, 512, 4096))
        return make_case(name=name, seed=2, seq_lens=ql, seq_lens_kv=kv,
                         q_heads=32, kv_heads=8, kv_dtype=INT8, scale_kind=PER_CHANNEL,
                         causal=True, chunk_size=512, num_pages=4096)
    if n == 3:
        bsz = 8
        return make_case(name="append-3", seed=3,
                         seq_lens=_draw_lens(3, S_LEN_Q, bsz, 64, 512),
                         seq_lens_kv=_draw_lens(3, S_LEN_KV, bsz, 0, 8192),
                         q_heads=32, kv_heads=8, kv_dtype=FP8, scale_kind=PER_HEAD,
                         causal=True, chunk_size=0)
    if n == 4:
        bsz = 128
        name, ql, kv = cut("spec-verify-4", np.full(bsz, 6, np.int32),
                           _draw_lens(4, S_LEN_KV, bsz, 8192, 32768))
        return make_case(name=name, seed=4, seq_lens=ql, seq_lens_kv=kv,
                         q_heads=64, kv_heads=8, kv_dtype=INT8, scale_kind=PER_HEAD,
                         causal=True, chunk_size=1024)
    if n == 5:
        bsz = 32
        name, ql, kv = cut("mla-5", _draw_lens(5, S_LEN_Q, bsz, 1, 2),
                           _draw_lens(5, S_LEN_KV, bsz, 4096, 16384))
        return make_case(name=name, seed=5, seq_lens=ql, seq_lens_kv=kv,
                         q_heads=128, kv_heads=1, head_dim_qk=576, head_dim_v=512,
                         kv_dtype=FP8, scale_kind=GLOBAL, layout=MLA, causal=True,
                         chunk_size=-1, sm_scale=1.0 / math.sqrt(192.0))
    raise ValueError(n)


def new_kv(case: Case):
    """bf16 keys / values of the appended tokens, to be quantised into the cache.

    GQA: (k [T, kv_heads, Dqk], v [T, kv_heads, Dv]) bf16 bit patterns; MLA:
    (k [T, Dqk], None).  Values are N(0, 1) times the stored-value spread of
    the cache: 40 x the channel's scale for int8 (so x / s mostly stays within
    +-127 and a few values saturate), 1 for fp8 (its scales map the N(0, 1)
    pool onto +-448).
    """
    T = case.total_q

    def draws(stream, shape, spread):
        n = int(np.prod(shape))
        x = rng.normal(case.seed, stream, np.arange(n, dtype=np.uint64)).reshape(shape)
        return to_bf16_bits(x * spread)

    def spread(which, heads, D):
        if case.kv_dtype == FP8:
            return 1.0
        sc = case.k_scale if which == "k" else case.v_scale
        if case.scale_kind == GLOBAL:
            return 40.0 * float(np.asarray(sc, np.float32).reshape(-1)[0])
        s = bf16_bits_to_f64(np.asarray(sc, np.uint16))
        if case.scale_kind == PER_HEAD:
            return 40.0 * s.reshape(heads, 1)
        return 40.0 * s.reshape(heads, D)

    if case.layout == MLA:
        return draws(S_KNEW, (T, case.head_dim_qk), spread("k", 1, case.head_dim_qk)), None
    k = draws(S_KNEW, (T, case.kv_heads, case.head_dim_qk),
              spread("k", case.kv_heads, case.head_dim_qk))
    v = draws(S_VNEW, (T, case.kv_heads, case.head_dim_v),
              spread("v", case.kv_heads, case.head_dim_v))
    return k, v


def tree_mask(case: Case) -> np.ndarray:
    """A seeded draft tree per sequence: appended token 0 is the root, token i
    > 0 hangs under a parent drawn uniformly from 0 .. i-1, and a token sees
    itself and its ancestors.  Returns uint8 [bsz, max_q, max_q]."""
    max_q = int(case.seq_lens.max()) if case.bsz else 0
    m = np.zeros((case.bsz, max_q, max_q), np.uint8)
    for b in range(case.bsz):
        n = int(case.seq_lens[b])
        for i in range(n):
            if i > 0:
                parent = int(rng.uniform_int(case.seed, S_TREE,
                                             np.array([b * 4096 + i], np.uint64), 0, i - 1)[0])
                m[b, i] = m[b, parent]
            m[b, i, i] = 1
    return m
