"""Pins for the oracle's planner: a hand-worked example of the written spec and
invariants any correct plan satisfies."""
import math

import numpy as np
import pytest

import synth
from oracle import planner as op


def _case(**kw):
    base = dict(name="p", seed=3, seq_lens=[3, 1], seq_lens_kv=[70, 0], q_heads=8,
                kv_heads=2, head_dim_qk=32, chunk_size=64, causal=True)
    base.update(kw)
    return synth.make_case(**base)


def test_hand_worked_example():
    """bsz 2, q_len [3,1], prefix [70,0], G 4, Hkv 2, causal, chunk 64, 3 SMs.

    decode family (3*4 <= 64), one tile per sequence; lim = 73 and 1; sequence 0
    splits into [0,64) and [64,73), sequence 1 has [0,1).  All six items cost 3,
    so the longest-first pass deals them round-robin over the 3 CTAs."""
    P = op.plan(_case(), num_sms=3)
    assert P["family"] == "decode" and P["chunk"] == 64 and P["num_ctas"] == 3
    s0 = lambda kvh, c: [0, kvh, 0, 3, 70, 64 * c, [64, 73][c], c | (2 << 16)]
    s1 = lambda kvh: [1, kvh, 3, 1, 0, 0, 1, 0 | (1 << 16)]
    want = [s0(0, 0), s0(1, 1), s0(0, 1), s1(0), s0(1, 0), s1(1)]
    assert P["items"].tolist() == want
    assert P["work_indptr"].tolist() == [0, 2, 4, 6]
    assert P["nch_token"].tolist() == [2, 2, 2, 1]
    assert P["max_chunks"] == 2 and P["merge_tokens"].tolist() == [0, 1, 2]


def _check_invariants(case, P):
    G = case.q_heads // case.kv_heads
    B = case.block_size
    items = P["items"]
    # each (token, kv head) sees chunks that partition [0, its tile limit)
    cover = {}
    for it in items.tolist():
        b, kvh, t0, nt, base, kv0, kv1, cc = it
        c, nch = cc & 0xFFFF, cc >> 16
        assert 0 <= kv0 < kv1 and c < nch
        cover.setdefault((b, kvh, t0), []).append((c, nch, kv0, kv1, nt, base))
    for (b, kvh, t0), lst in cover.items():
        lst.sort()
        nch = lst[0][1]
        assert [x[0] for x in lst] == list(range(nch))
        assert lst[0][2] == 0
        for x, y in zip(lst, lst[1:]):
            assert x[3] == y[2]
        nt, base = lst[0][4], lst[0][5]
        ql = int(case.seq_lens[b])
        tok0 = t0 - int(case.cu_seqlens_q[b])
        lim = (int(case.seq_lens_kv[b]) + tok0 + nt) if case.causal else (int(case.seq_lens_kv[b]) + ql)
        assert lst[-1][3] == lim
        if case.causal:
            assert base == int(case.seq_lens_kv[b]) + tok0
    # every query token is in exactly one tile per kv head
    T = case.total_q
    seen = np.zeros((T, case.kv_heads), int)
    for (b, kvh, t0), lst in cover.items():
        seen[t0:t0 + lst[0][4], kvh] += 1
    assert (seen == 1).all()
    # work lists
    ind = P["work_indptr"]
    assert ind[0] == 0 and ind[-1] == len(items) and (np.diff(ind) >= 1).all()
    # longest-first balance: max load - min load <= largest item cost
    cost = np.array([math.ceil((r[6] - r[5]) / B) + 2 for r in items.tolist()])
    loads = np.array([cost[ind[k]:ind[k + 1]].sum() for k in range(len(ind) - 1)])
    assert loads.max() - loads.min() <= cost.max()


@pytest.mark.parametrize("kw,sms", [
    (dict(), 3),
    (dict(causal=False, chunk_size=128), 5),
    (dict(seq_lens=[40, 0, 17], seq_lens_kv=[5, 9, 300], chunk_size=0), 7),     # append family
    (dict(seq_lens=[200], seq_lens_kv=[1000], q_heads=32, kv_heads=8, chunk_size=256), 152),
])
def test_plan_invariants(kw, sms):
    case = _case(**kw)
    P = op.plan(case, sms)
    _check_invariants(case, P)


def test_family_selection():
    assert op.plan(_case(seq_lens=[16, 1]), 4)["family"] == "decode"     # 16*4 = 64
    assert op.plan(_case(seq_lens=[17, 1]), 4)["family"] == "append"
    c5 = synth.make_case(seq_lens=[1, 2], seq_lens_kv=[4000, 9000], q_heads=128, kv_heads=1,
                         head_dim_qk=576, head_dim_v=512, kv_dtype="fp8_e4m3",
                         scale_kind="global", layout="mla", chunk_size=-1)
    P = op.plan(c5, 152)
    assert P["family"] == "mla" and P["tokens_per_tile"] == 1


def test_auto_chunk_rule():
    """chunk_size -1 (GQA): cs = max(4B, roundup(ceil(W / (4*slots)), B)) with W =
    kv_heads * sum of tile limits, no split when that reaches the longest limit."""
    c = synth.make_case(seq_lens=[1, 2], seq_lens_kv=[4000, 9000], q_heads=8, kv_heads=2,
                        chunk_size=-1)
    # one tile per sequence (16 tokens per tile at G = 4): limits 4001 and 9002
    W = 2 * (4001 + 9002)
    assert op.plan(c, 152)["chunk"] == max(256, math.ceil(math.ceil(W / 608) / 64) * 64) == 256
    assert op.plan(c, 2)["chunk"] == 3264       # ceil(26006 / 8) = 3251 -> 3264 < 9002
    assert op.plan(c, 1)["chunk"] == 6528       # ceil(26006 / 4) = 6502 -> 6528 < 9002
    big = synth.make_case(seq_lens=[1], seq_lens_kv=[100], q_heads=4, kv_heads=1,
                          chunk_size=-1)
    assert op.plan(big, 152)["chunk"] == 0      # 256 >= 101: no split


def test_mla_share_rule():
    """MLA, chunk_size -1: contiguous shares of all tiles' pages, worked by hand.
    Tiles (one token each): limits 4001, 9001, 9002 -> 63, 141, 141 pages,
    pages 0-62, 63-203, 204-344 (total 345).  152 SMs = 76 pairs: quota =
    max(4, ceil(345 / 76)) = 5, 69 pairs, pair k owns pages [5k, 5k + 5)."""
    c = synth.make_case(seq_lens=[1, 2], seq_lens_kv=[4000, 9000], q_heads=128, kv_heads=1,
                        head_dim_qk=576, head_dim_v=512, kv_dtype="fp8_e4m3",
                        scale_kind="global", layout="mla", chunk_size=-1)
    P = op.plan(c, 152)
    assert P["num_ctas"] == 69 and P["chunk"] == 320
    # pairs 0-12 touch token 0, 12-40 token 1, 40-68 token 2
    assert P["nch_token"].tolist() == [13, 29, 29] and P["max_chunks"] == 29
    ind, items = P["work_indptr"], P["items"]
    # pair 12: pages 60-64 = token 0's pages 60-62 and token 1's pages 0-1
    assert items[ind[12]:ind[13]].tolist() == [
        [0, 0, 0, 1, 4000, 3840, 4001, 12 | (13 << 16)],
        [1, 0, 1, 1, 9000, 0, 128, 0 | (29 << 16)]]
    # pair 68: token 2's last pages 340-344 -> local pages 136-140
    assert items[ind[68]:ind[69]].tolist() == [[1, 0, 2, 1, 9001, 136 * 64, 9002, 28 | (29 << 16)]]
    # every pair holds 5 pages
    pages = np.zeros(69, int)
    for k in range(69):
        for r in items[ind[k]:ind[k + 1]]:
            pages[k] += math.ceil(r[6] / 64) - r[5] // 64
    assert (pages == 5).all()
    # one pair: no split, the plain items
    P1 = op.plan(c, 2)
    assert P1["num_ctas"] == 1 and P1["chunk"] == 0 and P1["max_chunks"] == 1
    assert P1["items"][:, 5].tolist() == [0, 0, 0] and P1["items"][:, 6].tolist() == [4001, 9001, 9002]


def test_workload_truncation_keeps_the_same_draws():
    """A profiling capture's smaller case is the first sequences of the workload:
    the same lengths, hence the same per-sequence cache bytes."""
    full, part = synth.config(4), synth.config(4, 16)
    assert part.bsz == 16 and part.name.startswith("spec-verify-4")
    assert list(part.seq_lens) == list(full.seq_lens[:16])
    assert list(part.seq_lens_kv) == list(full.seq_lens_kv[:16])
    assert synth.config(2, 0).bsz == synth.config(2).bsz
