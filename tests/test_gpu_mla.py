"""GPU parity of the MLA path (128 query heads over one latent head, K 576 /
V 512, global scale) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import synth
from gpu_helpers import run_case, compare, reference_all

pytestmark = pytest.mark.gpu

MLA = dict(q_heads=128, kv_heads=1, head_dim_qk=576, head_dim_v=512, layout="mla",
           scale_kind="global", sm_scale=1.0 / np.sqrt(192.0))


def _mla_case(seed, **kw):
    args = dict(MLA)
    args.setdefault("kv_dtype", "fp8_e4m3")
    args.update(kw)
    return synth.make_case(name="mla-edge", seed=seed, **args)


EDGE = [
    # kv ranges around page boundaries, one token each, no split
    dict(seq_lens=[1, 1, 1, 1], seq_lens_kv=[0, 63, 64, 200], chunk_size=0),
    # two tokens (causal between them), split with merge
    dict(seq_lens=[2, 1, 2], seq_lens_kv=[700, 1000, 129], chunk_size=256),
    # planner's automatic chunk size
    dict(seq_lens=[1, 2], seq_lens_kv=[3000, 2500], chunk_size=-1),
    # int8 latent cache with a global scale
    dict(seq_lens=[2, 1], seq_lens_kv=[333, 64], chunk_size=128, kv_dtype="int8"),
    # non-causal
    dict(seq_lens=[2], seq_lens_kv=[190], chunk_size=0, causal=False),
]


@pytest.mark.parametrize("kw", EDGE)
def test_mla_edge_cases(kw):
    case = _mla_case(21, **kw)
    out, lse, plan, _, _ = run_case(case)
    assert plan.describe()["family"] == "mla"
    compare(case, out, lse, label=str(kw))


# the planner's contiguous page shares on a small grid: several short tokens
# share a pair, and shares cut tokens at page boundaries (8 SMs = 4 pairs;
# 11 pages -> shares of 4 pages), causal and not
SHARES = [
    dict(seq_lens=[1, 1, 1, 2, 1], seq_lens_kv=[10, 70, 0, 130, 5], chunk_size=-1),
    dict(seq_lens=[2, 1], seq_lens_kv=[300, 190], chunk_size=-1, causal=False),
]


@pytest.mark.parametrize("kw", SHARES)
def test_mla_page_shares(kw):
    case = _mla_case(23, **kw)
    out, lse, plan, _, _ = run_case(case, sms=8)
    d = plan.describe()
    assert d["family"] == "mla" and d["max_chunks"] > 1
    # every pair holds at most `quota` pages and the pieces of a token are in position order
    items, ind = d["items"], d["work_indptr"]
    for k in range(d["num_ctas"]):
        pages = sum(-(-int(r[6]) // 64) - int(r[5]) // 64 for r in items[ind[k]:ind[k + 1]])
        assert pages <= d["chunk"] // 64
    compare(case, out, lse, label=str(kw))


def test_mla_5_full():
    """Full-size MLA workload (bsz 32, q_len U{1,2}, prefix U[4096,16384], fp8
    global scale, automatic split + merge) in the benchmark's launch
    configuration; the oracle checks all 32 sequences."""
    case = synth.config(5)
    out, lse, plan, _, _ = run_case(case)
    d = plan.describe()
    assert d["family"] == "mla" and d["max_chunks"] > 1
    compare(case, out, lse, label="mla-5 (every sequence)", ref=reference_all(5, case))


def test_mla_repeat_bitexact():
    case = _mla_case(22, seq_lens=[2, 1], seq_lens_kv=[900, 50], chunk_size=256)
    out1, lse1, _, d, _ = run_case(case)
    out2, lse2, _, _, _ = run_case(case, d=d)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)
