"""Pins for the fp64 oracle: each check fixes the oracle to something other than
itself (closed forms, invariants of attention, a brute-force evaluation written
independently here, and library routines on special cases)."""
import math

import numpy as np
import pytest
import torch

import synth
from synth import cases as sc
from oracle import attention as oa
from oracle import formats as of


# --------------------------------------------------------------------------
# element formats
def test_e4m3_closed_forms():
    tab = of.decode_table("fp8_e4m3")
    assert tab[0x00] == 0.0 and math.copysign(1.0, tab[0x80]) == -1.0
    assert tab[0x01] == 2.0 ** -9           # smallest subnormal
    assert tab[0x07] == 7 * 2.0 ** -9       # largest subnormal
    assert tab[0x08] == 2.0 ** -6           # smallest normal
    assert tab[0x38] == 1.0
    assert tab[0x7E] == 448.0 and tab[0xFE] == -448.0   # the E4M3 maximum
    assert np.isnan(tab[0x7F]) and np.isnan(tab[0xFF])
    assert np.isnan(tab).sum() == 2


def test_e4m3_matches_library():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    tab = of.decode_table("fp8_e4m3")
    nan = np.isnan(lib)
    assert (nan == np.isnan(tab)).all()
    assert (lib[~nan] == tab[~nan]).all()


def test_int8_table_matches_twos_complement():
    tab = of.decode_table("int8")
    lib = np.arange(256, dtype=np.uint8).view(np.int8).astype(np.float64)
    assert (tab == lib).all()
    assert tab[0x7F] == 127 and tab[0x81] == -127 and tab[0x80] == -128


def test_bf16_decode_matches_library():
    bits = np.array([0x0000, 0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F, 0x3C23], np.uint16)
    lib = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert (of.bf16_to_f64(bits) == lib).all()


# --------------------------------------------------------------------------
# helpers: small cases and an independent brute-force evaluation
def small_case(**kw):
    base = dict(name="t", seed=11, seq_lens=[3, 1, 5], seq_lens_kv=[70, 0, 129],
                q_heads=8, kv_heads=2, head_dim_qk=32, kv_dtype="int8",
                scale_kind="per_kv_head", causal=True, chunk_size=0)
    base.update(kw)
    return synth.make_case(**base)


def brute(case):
    """Attention written element by element from the definition, with library
    decoders (numpy int8 view / torch float8) and torch softmax."""
    Hq, Hkv = case.q_heads, case.kv_heads
    G = Hq // Hkv
    D, Dv, B = case.head_dim_qk, case.head_dim_v, case.block_size
    if case.kv_dtype == "int8":
        dec = lambda a: np.asarray(a, np.uint8).view(np.int8).astype(np.float64)
    else:
        dec = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.uint8)).view(
            torch.float8_e4m3fn).to(torch.float64).numpy()
    bf = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()

    def sc_(which, kvh, dim):
        s = case.k_scale if which == "k" else case.v_scale
        if case.scale_kind == "per_kv_head":
            return np.full(dim, bf(s[kvh:kvh + 1])[0])
        if case.scale_kind == "per_channel":
            return bf(s[kvh * dim:(kvh + 1) * dim])
        return np.full(dim, float(s[0]))

    T = case.total_q
    out = np.zeros((T, Hq, Dv))
    lse = np.zeros((T, Hq))
    ck, cv = case.cache_k, case.cache_v
    for b in range(case.bsz):
        ql, pre = int(case.seq_lens[b]), int(case.seq_lens_kv[b])
        n = pre + ql
        for h in range(Hq):
            kvh = h // G
            ks = sc_("k", kvh, D)
            vs = sc_("v", kvh, Dv)
            K = np.zeros((n, D))
            V = np.zeros((n, Dv))
            for j in range(n):
                page = int(case.block_table[b, j // B])
                o = j % B
                if case.layout == "mla":
                    K[j] = dec(ck[page, o, :D]) * ks
                    V[j] = dec(ck[page, o, :Dv]) * vs
                else:
                    K[j] = dec(ck[page, kvh, o, :]) * ks
                    V[j] = dec(cv[page, kvh, :, o]) * vs
            for i in range(ql):
                t = int(case.cu_seqlens_q[b]) + i
                q = bf(case.q_bits[t, h * D:(h + 1) * D])
                mask = np.array([(not case.causal) or j <= pre + i for j in range(n)])
                if case.attn_mask is not None:   # draft tree: ancestors among appended tokens
                    mask &= np.array([j < pre or bool(case.attn_mask[b, i, j - pre])
                                      for j in range(n)])
                s = torch.from_numpy(case.sm_scale * (K @ q))
                s[~torch.from_numpy(mask)] = -torch.inf
                w = torch.softmax(s, dim=0).numpy()
                out[t, h] = w @ V
                lse[t, h] = torch.logsumexp(s, dim=0).item()
    return out, lse


@pytest.mark.parametrize("kw", [
    dict(),
    dict(causal=False),
    dict(scale_kind="per_channel"),
    dict(kv_dtype="fp8_e4m3", seq_lens=[2, 4], seq_lens_kv=[10, 64]),
    dict(q_heads=4, kv_heads=4, seq_lens=[2, 3], seq_lens_kv=[5, 63]),
    dict(layout="mla", q_heads=4, kv_heads=1, head_dim_qk=40, head_dim_v=32,
         kv_dtype="fp8_e4m3", scale_kind="global", seq_lens=[1, 2], seq_lens_kv=[65, 3]),
    dict(q_stride=8 * 32 + 2 * 2 * 32),   # packed qkv row stride
])
def test_brute_force_agrees(kw):
    """I4: an independent dense evaluation matches to 1e-12."""
    case = small_case(**kw)
    out, lse = oa.reference(case)
    bo, bl = brute(case)
    assert np.allclose(out, bo, rtol=0, atol=1e-12)
    assert np.allclose(lse, bl, rtol=0, atol=1e-12)


def test_single_key_returns_v():
    """I1: one visible key gives out = v exactly and lse = s."""
    case = small_case(seq_lens=[1], seq_lens_kv=[0], q_heads=4, kv_heads=1)
    out, lse = oa.reference(case)
    K, V = oa.dequant_kv(case, 0, 0, 1)
    q = oa.q_rows(case, 0, 0)[0]             # [G, D]
    for g in range(4):
        assert (out[0, g] == V[0]).all()
        assert lse[0, g] == pytest.approx(case.sm_scale * float(q[g] @ K[0]), abs=1e-14)


def test_identical_keys_average_v():
    """I2: n identical keys give the mean of V and lse = s + ln n."""
    case = small_case(seq_lens=[1], seq_lens_kv=[99], q_heads=2, kv_heads=1, causal=False)
    ck = case.cache_k.copy()
    ck[:, :, :, :] = ck[0, 0, 0, :]          # every K row equal
    case._cache_k = ck
    out, lse = oa.reference(case)
    K, V = oa.dequant_kv(case, 0, 0, 100)
    q = oa.q_rows(case, 0, 0)[0]
    for g in range(2):
        assert np.allclose(out[0, g], V.mean(axis=0), atol=1e-13, rtol=0)
        s = case.sm_scale * float(q[g] @ K[0])
        assert lse[0, g] == pytest.approx(s + math.log(100), abs=1e-12)


@pytest.mark.parametrize("chunk", [1, 7, 64, 100, 128, 10_000])
def test_split_merge_equals_unsplit(chunk):
    """I3: per-chunk states merged by log-sum-exp equal unsplit attention."""
    case = small_case()
    out, lse = oa.reference(case)
    so, sl = oa.reference_split(case, chunk)
    assert np.allclose(out, so, atol=1e-12, rtol=0)
    assert np.allclose(lse, sl, atol=1e-12, rtol=0)


def test_empty_chunk_state_is_neutral():
    """A chunk with no visible position (m = -inf, d = 0) leaves the merge unchanged."""
    case = small_case(seq_lens=[4], seq_lens_kv=[8], q_heads=2, kv_heads=1)
    bounds = [(0, 5), (5, 12)]
    M, Dn, O = oa.unit_partials(case, 0, 0, bounds)
    # token 0 sees j <= 8: chunk (9, 12) is empty for it
    M2, D2, O2 = oa.unit_partials(case, 0, 0, bounds + [(9, 12)])
    assert np.isneginf(M2[2, 0]).all() and (D2[2, 0] == 0).all()
    o1, l1 = oa.merge_states(M, Dn, O)
    o2, l2 = oa.merge_states(M2[:2], D2[:2], O2[:2])
    assert np.allclose(o1, o2) and np.allclose(l1, l2)


def test_page_permutation_invariance():
    """I5: relabelling physical pages (pool and block table together) changes nothing."""
    case = small_case()
    out, lse = oa.reference(case)
    P = case.num_pages
    perm = np.random.default_rng(0).permutation(P)
    inv = np.argsort(perm)
    c2 = small_case()
    c2._cache_k = case.cache_k[inv]          # new page p holds old page inv[p]
    c2._cache_v = case.cache_v[inv]
    bt = case.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    c2.block_table = bt
    o2, l2 = oa.reference(c2)
    assert (out == o2).all() and (lse == l2).all()


def test_per_channel_equal_scales_reproduce_per_head():
    """I6: per-channel scales all equal to c reproduce the per-head scale c."""
    a = small_case(scale_kind="per_kv_head")
    b = small_case(scale_kind="per_channel")
    b.k_scale = np.repeat(a.k_scale, 32)
    b.v_scale = np.repeat(a.v_scale, 32)
    oa_, la = oa.reference(a)
    ob, lb = oa.reference(b)
    assert np.allclose(oa_, ob, atol=1e-14) and np.allclose(la, lb, atol=1e-14)


def test_mha_noncausal_is_textbook_sdpa():
    """I7: G = 1 with a non-causal full prefix is scaled-dot-product attention."""
    case = small_case(q_heads=3, kv_heads=3, seq_lens=[4], seq_lens_kv=[60], causal=False)
    out, _ = oa.reference(case)
    qs, ks, vs = [], [], []
    for h in range(3):
        K, V = oa.dequant_kv(case, 0, h, 64)
        qs.append(oa.q_rows(case, 0, h)[:, 0, :])
        ks.append(K)
        vs.append(V)
    Q = torch.from_numpy(np.stack(qs))
    K = torch.from_numpy(np.stack(ks))
    V = torch.from_numpy(np.stack(vs))
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=case.sm_scale)
    assert np.allclose(out[:, :, :], ref.permute(1, 0, 2).numpy(), atol=1e-12, rtol=0)


def test_lse_normalises():
    """I8: sum_j exp(s_j - lse) = 1 over the visible positions."""
    case = small_case()
    _, lse = oa.reference(case)
    G = case.group
    for b in range(case.bsz):
        for kvh in range(case.kv_heads):
            S, V, n = oa.unit_scores(case, b, kvh)
            ql = S.shape[0]
            for i in range(ql):
                t = int(case.cu_seqlens_q[b]) + i
                for g in range(G):
                    vis = np.arange(n) <= int(case.seq_lens_kv[b]) + i
                    z = np.exp(S[i, g, vis] - lse[t, kvh * G + g]).sum()
                    assert z == pytest.approx(1.0, abs=1e-12)


def test_causal_bound_is_inclusive_of_own_position():
    """The appended token i sees position seq_lens_kv + i (its own K/V) and not i + 1."""
    case = small_case(seq_lens=[3], seq_lens_kv=[5], q_heads=1, kv_heads=1, head_dim_qk=32)
    S, V, n = oa.unit_scores(case, 0, 0)
    vis = oa._visible(case, 0, 3, n, 0, n)
    assert vis[0].tolist() == [True] * 6 + [False] * 2
    assert vis[2].tolist() == [True] * 8


def test_lazy_pages_match_materialised_pool():
    """Page regeneration from counters equals the materialised pool."""
    case = small_case()
    for p in range(case.num_pages):
        assert (case.page_k(p) == case.cache_k[p]).all()
        assert (case.page_v(p) == case.cache_v[p]).all()


def test_workload_shapes():
    """The five workloads have the stated shapes and draws in range."""
    c1 = synth.config(1)
    assert c1.seq_lens_kv.tolist() == [100, 37] and c1.block_table.shape == (2, 4)
    assert sorted(c1.block_table.reshape(-1).tolist()) == list(range(8))
    c2 = synth.config(2)
    assert c2.num_pages == 4096 and c2.k_scale.shape == (8 * 128,)
    assert c2.seq_lens_kv.min() >= 512 and c2.seq_lens_kv.max() <= 4096
    assert (np.ceil(c2.kvtot / 64).sum()) <= 4096
    c4 = synth.config(4)
    assert (c4.seq_lens == 6).all() and c4.q_heads == 64 and c4.chunk_size == 1024
    assert c4.seq_lens_kv.min() >= 8192 and c4.seq_lens_kv.max() <= 32768


def _with_mask(case, mask):
    case.attn_mask = mask
    return case


def test_tree_mask_brute_force_agrees():
    """The draft-tree visibility rule against the element-by-element evaluation."""
    from synth.cases import tree_mask
    case = small_case(seq_lens=[6, 1, 5], seq_lens_kv=[70, 0, 129])
    _with_mask(case, tree_mask(case))
    assert case.attn_mask[0].sum() > 6 and not np.all(np.tril(case.attn_mask[0]) == 1)
    out, lse = oa.reference(case)
    bo, bl = brute(case)
    assert np.allclose(out, bo, rtol=0, atol=1e-12)
    assert np.allclose(lse, bl, rtol=0, atol=1e-12)


def test_full_lower_triangular_tree_is_causal():
    """A chain (every token sees all earlier draft tokens) is plain causal."""
    case = small_case(seq_lens=[6, 3], seq_lens_kv=[40, 64])
    o1, l1 = oa.reference(case)
    _with_mask(case, np.tril(np.ones((2, 6, 6), np.uint8)))
    o2, l2 = oa.reference(case)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_root_only_tree_sees_prefix_and_itself():
    """With no edges, token i attends over the prefix and its own position only:
    the same as a single-token decode at position seq_lens_kv + i."""
    case = small_case(seq_lens=[4], seq_lens_kv=[100])
    _with_mask(case, np.eye(4, dtype=np.uint8)[None])
    out, lse = oa.reference(case)
    S, V, kvtot = oa.unit_scores(case, 0, 0)
    G = case.q_heads // case.kv_heads
    for i in range(4):
        idx = np.r_[np.arange(100), 100 + i]
        s = S[i, :, idx].T                      # [G, n]
        m = s.max(axis=1, keepdims=True)
        w = np.exp(s - m)
        ref = (w @ V[idx]) / w.sum(axis=1, keepdims=True)
        assert np.allclose(out[i, :G], ref, rtol=0, atol=1e-12)
