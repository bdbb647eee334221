"""CPU checks of the C ABI: the library loads, exports every declared entry
point, validates arguments before any launch, and its planner reproduces the
oracle planner bit for bit."""
import os
import re

import numpy as np
import pytest

import synth
from oracle import planner as op

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pa():
    import paged_quantized_kv_gqa_gb300 as m
    return m


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(pa):
    names = declared_functions()
    assert "pa_plan" in names and "pa_run" in names and "pa_merge" in names
    for n in names:
        assert hasattr(pa.lib, n), n


def _plan(pa, case, sms=152):
    return pa.pa_plan(pa.problem_of(case), case.seq_lens, case.seq_lens_kv, case.cu_seqlens_q, sms)


CASES = [
    dict(seq_lens=[3, 1], seq_lens_kv=[70, 0], q_heads=8, kv_heads=2, chunk_size=64),
    dict(seq_lens=[1] * 9, seq_lens_kv=list(range(0, 900, 100)), q_heads=32, kv_heads=8,
         chunk_size=128, causal=False),
    dict(seq_lens=[40, 0, 17], seq_lens_kv=[5, 9, 300], q_heads=8, kv_heads=2, chunk_size=0),
    dict(seq_lens=[200, 3], seq_lens_kv=[1000, 4000], q_heads=32, kv_heads=8, chunk_size=256),
    dict(seq_lens=[6] * 5, seq_lens_kv=[8000, 9000, 100, 64, 63], q_heads=64, kv_heads=8,
         chunk_size=1024),
    dict(seq_lens=[1, 2, 2], seq_lens_kv=[4000, 9000, 17], q_heads=128, kv_heads=1,
         head_dim_qk=576, head_dim_v=512, kv_dtype="fp8_e4m3", scale_kind="global",
         layout="mla", chunk_size=-1),
    dict(seq_lens=[5, 7], seq_lens_kv=[3000, 10], q_heads=16, kv_heads=4, chunk_size=-1),
]


@pytest.mark.parametrize("kw", CASES)
@pytest.mark.parametrize("sms", [1, 7, 152])
def test_planner_matches_oracle(pa, kw, sms):
    case = synth.make_case(name="p", seed=5, **kw)
    got = _plan(pa, case, sms).describe()
    want = op.plan(case, sms)
    for key in ("family", "chunk", "tokens_per_tile", "num_ctas", "max_chunks"):
        assert got[key] == want[key], key
    for key in ("items", "work_indptr", "nch_token", "merge_tokens"):
        assert np.array_equal(got[key], want[key]), key


def _random_problem(r):
    """A seeded random problem of one of the three families: lengths with
    zeros, ragged query counts, every chunk rule, causal or not."""
    fam = r.choice(["decode", "append", "mla"])
    bsz = int(r.integers(1, 9))
    if fam == "mla":
        kw = dict(q_heads=128, kv_heads=1, head_dim_qk=576, head_dim_v=512, kv_dtype="fp8_e4m3",
                  scale_kind="global", layout="mla")
        q = r.integers(1, 3, bsz)
    else:
        kvh = int(r.choice([1, 2, 4, 8]))
        kw = dict(q_heads=kvh * int(r.choice([1, 2, 4, 8])), kv_heads=kvh)
        q = r.integers(0, 5, bsz) if fam == "decode" else r.integers(0, 200, bsz)
    q[int(r.integers(0, bsz))] = max(1, int(q.max()))    # at least one query token
    kv = r.integers(0, 6000, bsz)
    kv[r.random(bsz) < 0.2] = 0
    kw.update(seq_lens=q.tolist(), seq_lens_kv=kv.tolist(), causal=bool(r.random() < 0.8),
              chunk_size=int(r.choice([0, 64, 128, 512, 1024, -1])))
    return kw


@pytest.mark.parametrize("seed", range(40))
def test_planner_matches_oracle_random(pa, seed):
    r = np.random.default_rng(1000 + seed)
    kw = _random_problem(r)
    sms = int(r.choice([1, 3, 8, 152]))
    case = synth.make_case(name="p", seed=seed, **kw)
    got = _plan(pa, case, sms).describe()
    want = op.plan(case, sms)
    for key in ("family", "chunk", "tokens_per_tile", "num_ctas", "max_chunks"):
        assert got[key] == want[key], (key, kw, sms)
    for key in ("items", "work_indptr", "nch_token", "merge_tokens"):
        assert np.array_equal(got[key], want[key]), (key, kw, sms)


@pytest.mark.parametrize("seed", range(12))
def test_plan_work_counts_match_the_oracle_mask(pa, seed):
    """The plan's flops (the numerator of the append / MLA TFLOP/s figures) are
    2 (Dqk + Dv) per visible (query head, position) pair: counted here from
    the oracle's own visibility mask; kv_bytes are the whole pages the
    sequences occupy."""
    from oracle.attention import _visible
    r = np.random.default_rng(2000 + seed)
    kw = _random_problem(r)
    case = synth.make_case(name="w", seed=seed, **kw)
    d = _plan(pa, case, 152).describe()
    pairs = 0
    pages = 0
    for b in range(len(case.seq_lens)):
        q, kvtot = int(case.seq_lens[b]), int(case.seq_lens_kv[b]) + int(case.seq_lens[b])
        if q == 0:
            continue
        pairs += int(_visible(case, b, q, kvtot, 0, kvtot).sum())
        pages += -(-kvtot // 64)
    per_pair = case.q_heads * 2 * (case.head_dim_qk + case.head_dim_v)
    assert d["flops"] == pairs * per_pair, kw
    row = case.head_dim_qk if case.layout == "mla" else (case.head_dim_qk + case.head_dim_v) * case.kv_heads
    assert d["kv_bytes"] == pages * 64 * row, kw


@pytest.mark.parametrize("seed", range(12))
def test_bench_kv_bytes_are_the_visible_rows_read_once(seed):
    """bench.py's GB/s numerator: every (sequence, kv head) reads the K and V
    rows of the positions any of its query tokens sees, once (MLA: the
    576-byte latent row, V being its prefix), counted from the oracle mask."""
    import bench
    from oracle.attention import _visible
    r = np.random.default_rng(3000 + seed)
    case = synth.make_case(name="w", seed=seed, **_random_problem(r))
    rows = 0
    for b in range(len(case.seq_lens)):
        q, kvtot = int(case.seq_lens[b]), int(case.seq_lens_kv[b]) + int(case.seq_lens[b])
        if q == 0:
            continue
        rows += int(_visible(case, b, q, kvtot, 0, kvtot).any(axis=0).sum())
    per_row = case.head_dim_qk if case.layout == "mla" else (case.head_dim_qk + case.head_dim_v) * case.kv_heads
    assert bench.algorithmic_bytes(case) == rows * per_row


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_planner_matches_oracle_on_workloads(pa, n):
    case = synth.config(n) if n != 3 and n != 5 else _light(n)
    got = _plan(pa, case, 152).describe()
    want = op.plan(case, 152)
    for key in ("family", "chunk", "num_ctas", "max_chunks"):
        assert got[key] == want[key], key
    for key in ("items", "work_indptr", "nch_token", "merge_tokens"):
        assert np.array_equal(got[key], want[key]), key


def _light(n):
    """Workloads 3 / 5 with their lengths and shapes but a tiny stand-in cache
    (the planner only reads lengths)."""
    full = {3: dict(q_heads=32, kv_heads=8, kv_dtype="int8", chunk_size=0),
            5: dict(q_heads=128, kv_heads=1, head_dim_qk=576, head_dim_v=512, kv_dtype="int8",
                    scale_kind="global", layout="mla", chunk_size=-1)}[n]
    from synth.cases import _draw_lens, S_LEN_Q, S_LEN_KV
    if n == 3:
        ql, kv = _draw_lens(3, S_LEN_Q, 8, 64, 512), _draw_lens(3, S_LEN_KV, 8, 0, 8192)
    else:
        ql, kv = _draw_lens(5, S_LEN_Q, 32, 1, 2), _draw_lens(5, S_LEN_KV, 32, 4096, 16384)
    return synth.make_case(name=f"light{n}", seed=n, seq_lens=ql, seq_lens_kv=kv, **full)


def test_workspace_and_work_counts(pa):
    case = synth.config(2)
    d = _plan(pa, case).describe()
    assert d["family"] == "decode" and d["chunk"] == 512
    assert d["kv_bytes"] == case.kv_bytes_total()
    T, H = case.total_q, case.q_heads
    assert d["workspace_bytes"] >= T * d["max_chunks"] * H * (128 * 2 + 8)


def test_fused_merge_only_for_split_decode_plans(pa):
    """With the single-launch option on, decode-family plans with split rows
    merge inside the attention launch; append / MLA plans and unsplit plans
    never do, and the option is off by default."""
    assert not _plan(pa, synth.config(2)).describe()["fused_merge"]     # default off
    pa.pa_set_fused_merge(True)
    try:
        assert _plan(pa, synth.config(2)).describe()["fused_merge"]
        assert _plan(pa, synth.config(4)).describe()["fused_merge"]
        assert not _plan(pa, synth.config(1)).describe()["fused_merge"]     # no split
        assert not _plan(pa, synth.config(3)).describe()["fused_merge"]     # append
        assert not _plan(pa, synth.config(5)).describe()["fused_merge"]     # MLA
    finally:
        pa.pa_set_fused_merge(False)
    assert not _plan(pa, synth.config(2)).describe()["fused_merge"]


@pytest.mark.parametrize("field,value,status", [
    ("chunk_size", 100, 1),        # not a multiple of the page size
    ("q_heads", 30, 1),            # not a multiple of kv_heads
    ("head_dim_qk", 64, 2),        # no kernel built for it
    ("sm_scale", -1.0, 1),
    ("q_stride", 12, 1),
])
def test_invalid_problems_rejected(pa, field, value, status):
    case = synth.make_case(name="v", seed=1, seq_lens=[2], seq_lens_kv=[10], q_heads=8,
                           kv_heads=2, chunk_size=0)
    prob = pa.problem_of(case)
    setattr(prob, field, value)
    with pytest.raises(pa.PaError) as e:
        pa.pa_plan(prob, case.seq_lens, case.seq_lens_kv, case.cu_seqlens_q, 152)
    assert e.value.status == status


def test_invalid_lengths_rejected(pa):
    case = synth.make_case(name="v", seed=1, seq_lens=[2, 3], seq_lens_kv=[10, 5], q_heads=8,
                           kv_heads=2, chunk_size=0)
    prob = pa.problem_of(case)
    with pytest.raises(pa.PaError):
        pa.pa_plan(prob, [2, -1], case.seq_lens_kv, [0, 2, 1], 152)
    with pytest.raises(pa.PaError):
        pa.pa_plan(prob, case.seq_lens, case.seq_lens_kv, [0, 2, 4], 152)   # not a prefix sum
    with pytest.raises(pa.PaError):
        pa.pa_plan(prob, case.seq_lens, [10, 10_000], case.cu_seqlens_q, 152)  # too many pages


def test_run_rejects_null_pointers_before_launch(pa):
    case = synth.make_case(name="v", seed=1, seq_lens=[1], seq_lens_kv=[10], q_heads=8,
                           kv_heads=2, chunk_size=0)
    plan = _plan(pa, case)
    args = pa.make_args(q=None, cache_k=None, cache_v=None, k_scale=None, v_scale=None,
                        block_table=None, out=16)
    with pytest.raises(pa.PaError) as e:
        pa.pa_run(plan, args, 256, None)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    with pytest.raises(pa.PaError) as e:
        pa.pa_run(plan, args, None, None)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    args2 = pa.make_args(q=16, cache_k=32, cache_v=64, k_scale=8, v_scale=8, block_table=8,
                         out=8)
    args2.q = 18   # misaligned
    with pytest.raises(pa.PaError) as e:
        pa.pa_run(plan, args2, 256, None)
    assert e.value.status == pa.PA_ERR_INVALID_ARG


def test_default_library_has_no_pipeline_trace(pa):
    """The pipeline trace exists only in the library built with PA_TRACE: the
    default one refuses a trace buffer (host-side check, no GPU needed) and
    accepts turning the trace off."""
    import ctypes
    assert pa.lib.pa_debug_set_trace(ctypes.c_void_p(256), 1, 1) == pa.PA_ERR_UNSUPPORTED
    assert "PA_TRACE" in pa.pa_last_error()
    assert pa.lib.pa_debug_set_trace(None, 0, 0) == pa.PA_OK
