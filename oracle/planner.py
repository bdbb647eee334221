"""Independent restatement of the work-item planner (oracle side).

The production planner (C++, behind pa_plan) must produce exactly these
arrays.  The spec comes from the way the source pages carve the grid:
FastDeploy append_attention_c8_impl.cuh (batch_ids / tile_ids_per_batch: one
CTA row per (sequence, q tile of packed (token, head-in-group) rows); chunk c
covers [c*chunk_size, min(kv_len, (c+1)*chunk_size)); the causal iteration
bound uses the tile's last token), FlashInfer persistent.cuh (a work list per
CTA, work_indptr, kv_start/kv_end per item) and XQA mla_sm120.cu (the sub-
sequence split sized from the SM count).

Spec:
  G = q_heads / kv_heads.  family = "mla" for the MLA layout; otherwise
  "decode" when max(q_len) * G <= 64, else "append".
  rows_cap = 64 (decode), 256 (append: two 128-row query tiles), q_heads
  (mla); tokens per tile tpt = rows_cap // G.  CTAs per item: 2 for mla, else 1; slots = num_sms //
  (CTAs per item).
  Tiles, sequence-major: for b, for t in 0..ceil(q_len_b / tpt)-1:
      tok0 = t*tpt, tok1 = min(q_len_b, tok0 + tpt),
      lim  = seq_lens_kv[b] + tok1 if causal else seq_lens_kv[b] + q_len_b.
  Chunk size cs: chunk_size > 0 -> cs; 0 -> no split; -1 (auto) ->
      W = kv_heads * sum(lim over tiles), cs = max(4*B, roundup(ceil(W / (4*slots)), B)),
      and no split when cs >= max lim.
  Items, in order: for each tile, for kvh, for c in 0..nch-1 with
      nch = 1 (no split) or ceil(lim / cs),
      kv0 = c*cs, kv1 = min(lim, kv0 + cs)  (no split: 0 .. lim).
  Item record (8 x int32): b, kvh, cu_seqlens_q[b] + tok0, tok1 - tok0,
      causal_base (seq_lens_kv[b] + tok0 if causal else kvtot_b), kv0, kv1,
      c | (nch << 16).   Query token tok0 + i of the tile sees positions
      j <= causal_base + i.
  cost = ceil((kv1 - kv0) / B) + 2.  num_ctas = min(#items, slots).
  Longest-first assignment: visit items by (cost descending, index ascending);
  give each to the CTA with the smallest accumulated cost (ties: lowest CTA);
  each CTA runs its items in the order received.  Items are stored CTA-major
  with work_indptr[num_ctas + 1].
  nch_token[t] = nch of token t's tile; max_chunks = max(1, max nch_token);
  merge_tokens = tokens with nch_token > 1, ascending.
  MLA with chunk_size = -1 replaces the chunk size and the longest-first
  deal by contiguous shares (this library's scheduling choice; the pages fix
  only what an item computes): the tiles' pages, ceil(lim / B) per tile,
  are numbered consecutively in tile order; quota = max(4, ceil(total /
  slots)); num_ctas = ceil(total / quota); CTA pair k owns pages [k*quota,
  min(total, (k+1)*quota)).  For each k, for each tile overlapping that
  range (tile order), one item covers the overlap: kv0 = (first overlapping
  page - the tile's first page) * B, kv1 = min(lim, (end of overlap - the
  tile's first page) * B), chunk index = how many pieces of that tile came
  before it, nch = the number of pairs overlapping the tile.  chunk (as
  reported) = quota * B if some tile has nch > 1, else 0.
"""
from __future__ import annotations

import heapq
import math

import numpy as np

DECODE_ROWS = 64
APPEND_ROWS = 256


def plan(p, num_sms: int) -> dict:
    bsz = len(p.seq_lens)
    G = p.q_heads // p.kv_heads
    B = p.block_size
    q_lens = [int(x) for x in p.seq_lens]
    slkv = [int(x) for x in p.seq_lens_kv]
    cu = [int(x) for x in p.cu_seqlens_q]
    max_q = max(q_lens) if bsz else 0
    if p.layout == "mla":
        family, rows_cap, per_item = "mla", p.q_heads, 2
    elif max_q * G <= DECODE_ROWS:
        family, rows_cap, per_item = "decode", DECODE_ROWS, 1
    else:
        family, rows_cap, per_item = "append", APPEND_ROWS, 1
    tpt = rows_cap // G
    slots = max(1, num_sms // per_item)

    tiles = []
    for b in range(bsz):
        ql = q_lens[b]
        for t in range(math.ceil(ql / tpt)):
            tok0 = t * tpt
            tok1 = min(ql, tok0 + tpt)
            lim = slkv[b] + tok1 if p.causal else slkv[b] + ql
            tiles.append((b, tok0, tok1, lim))

    if family == "mla" and int(p.chunk_size) == -1:
        return _mla_shares(p, tiles, slots, tpt, q_lens, slkv, cu, B)

    cs = int(p.chunk_size)
    if cs == -1:
        W = p.kv_heads * sum(t[3] for t in tiles)
        target = 4 * slots
        cs = max(4 * B, math.ceil(math.ceil(W / target) / B) * B) if tiles else 0
        if tiles and cs >= max(t[3] for t in tiles):
            cs = 0
    split = cs > 0

    items = []
    T = cu[-1] if cu else 0
    nch_token = np.zeros(T, dtype=np.int32)
    for (b, tok0, tok1, lim) in tiles:
        nch = math.ceil(lim / cs) if split else 1
        base = slkv[b] + tok0 if p.causal else slkv[b] + q_lens[b]
        nch_token[cu[b] + tok0:cu[b] + tok1] = nch
        for kvh in range(p.kv_heads):
            for c in range(nch):
                kv0 = c * cs if split else 0
                kv1 = min(lim, kv0 + cs) if split else lim
                items.append((b, kvh, cu[b] + tok0, tok1 - tok0, base, kv0, kv1, c | (nch << 16)))

    n = len(items)
    num_ctas = min(n, slots)
    cost = [math.ceil((it[6] - it[5]) / B) + 2 for it in items]
    order = sorted(range(n), key=lambda i: (-cost[i], i))
    heap = [(0, k) for k in range(num_ctas)]
    per_cta = [[] for _ in range(num_ctas)]
    for i in order:
        load, k = heapq.heappop(heap)
        per_cta[k].append(i)
        heapq.heappush(heap, (load + cost[i], k))
    indptr = np.zeros(num_ctas + 1, dtype=np.int32)
    flat = []
    for k in range(num_ctas):
        flat.extend(per_cta[k])
        indptr[k + 1] = len(flat)
    arr = np.array([items[i] for i in flat], dtype=np.int64).reshape(-1, 8).astype(np.int32)
    max_chunks = int(max(1, nch_token.max() if T else 1))
    merge_tokens = np.nonzero(nch_token > 1)[0].astype(np.int32)
    return dict(family=family, chunk=cs, tokens_per_tile=tpt, num_ctas=num_ctas,
                items=arr, work_indptr=indptr, nch_token=nch_token,
                max_chunks=max_chunks, merge_tokens=merge_tokens)


def _mla_shares(p, tiles, slots, tpt, q_lens, slkv, cu, B):
    """Contiguous shares of all tiles' pages (the MLA rule in the spec above)."""
    npages = [math.ceil(lim / B) for (_, _, _, lim) in tiles]
    start = [sum(npages[:i]) for i in range(len(tiles))]       # first page of each tile
    total = sum(npages)
    quota = max(4, math.ceil(total / slots))
    num_ctas = math.ceil(total / quota)
    owners = [[k for k in range(num_ctas)
               if start[i] < min(total, (k + 1) * quota) and start[i] + npages[i] > k * quota]
              for i in range(len(tiles))]
    T = cu[-1] if cu else 0
    nch_token = np.zeros(T, dtype=np.int32)
    for i, (b, tok0, tok1, lim) in enumerate(tiles):
        nch_token[cu[b] + tok0:cu[b] + tok1] = len(owners[i])
    rows = []
    indptr = np.zeros(num_ctas + 1, dtype=np.int32)
    for k in range(num_ctas):
        lo, hi = k * quota, min(total, (k + 1) * quota)
        for i, (b, tok0, tok1, lim) in enumerate(tiles):
            if k not in owners[i]:
                continue
            first = max(lo, start[i]) - start[i]
            last = min(hi, start[i] + npages[i]) - start[i]
            base = slkv[b] + tok0 if p.causal else slkv[b] + q_lens[b]
            c = owners[i].index(k)
            rows.append((b, 0, cu[b] + tok0, tok1 - tok0, base, first * B, min(lim, last * B),
                         c | (len(owners[i]) << 16)))
        indptr[k + 1] = len(rows)
    arr = np.array(rows, dtype=np.int64).reshape(-1, 8).astype(np.int32)
    split = bool(T) and int(nch_token.max()) > 1
    max_chunks = int(max(1, nch_token.max() if T else 1))
    merge_tokens = np.nonzero(nch_token > 1)[0].astype(np.int32)
    return dict(family="mla", chunk=quota * B if split else 0, tokens_per_tile=tpt,
                num_ctas=num_ctas, items=arr, work_indptr=indptr, nch_token=nch_token,
                max_chunks=max_chunks, merge_tokens=merge_tokens)
