"""GPU parity of the append (chunked-prefill) path, q_len * G > 64, against the
fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import synth
from gpu_helpers import run_case, compare, reference_all

pytestmark = pytest.mark.gpu


def test_append_3_full():
    """Full-size append workload (8 sequences, q_len U[64,512], prefix U[0,8192],
    fp8 per-head scales, causal) in the benchmark's launch configuration; the
    oracle checks every (sequence, kv head) unit."""
    case = synth.config(3)
    out, lse, plan, _, _ = run_case(case)
    d = plan.describe()
    assert d["family"] == "append" and d["chunk"] == 0
    compare(case, out, lse, label="append-3 (every unit)", ref=reference_all(3, case))


EDGE = [
    # ragged query runs: one tile, a partial second tile, several tiles
    dict(seq_lens=[17, 64, 100], seq_lens_kv=[0, 130, 1000], q_heads=32, kv_heads=8),
    # kv ranges that end on and around page / tile boundaries
    dict(seq_lens=[20, 20, 20, 20], seq_lens_kv=[44, 108, 109, 236], q_heads=32, kv_heads=8),
    # G = 1 (MHA), 256 tokens per item, non-causal
    dict(seq_lens=[300, 70], seq_lens_kv=[50, 900], q_heads=4, kv_heads=4, causal=False),
    # G = 8, int8 per-channel scales
    dict(seq_lens=[40, 9], seq_lens_kv=[600, 3], q_heads=64, kv_heads=8, scale_kind="per_channel"),
    # fp8 with one global scale
    dict(seq_lens=[33, 90], seq_lens_kv=[257, 0], q_heads=16, kv_heads=4, kv_dtype="fp8_e4m3",
         scale_kind="global"),
    # split kv chunks plus merge, causal rows that see nothing in late chunks
    dict(seq_lens=[130, 64], seq_lens_kv=[0, 700], q_heads=32, kv_heads=8, chunk_size=128),
    dict(seq_lens=[200], seq_lens_kv=[2000], q_heads=16, kv_heads=2, kv_dtype="fp8_e4m3",
         chunk_size=512),
    # packed qkv row stride, and a group that does not divide 256 (G = 3)
    dict(seq_lens=[50], seq_lens_kv=[300], q_heads=8, kv_heads=2, q_stride=(8 + 2 * 2) * 128),
    dict(seq_lens=[90, 30], seq_lens_kv=[77, 500], q_heads=6, kv_heads=2),
    # fewer query tokens in the whole batch than one item holds
    dict(seq_lens=[20], seq_lens_kv=[64], q_heads=32, kv_heads=8),
    # empty sequences mixed in
    dict(seq_lens=[0, 80, 0], seq_lens_kv=[10, 64, 0], q_heads=32, kv_heads=8),
]


@pytest.mark.parametrize("kw", EDGE)
def test_append_edge_cases(kw):
    kw = dict(kw)
    case = synth.make_case(name="edge", seed=11, **kw)
    out, lse, plan, _, _ = run_case(case)
    assert plan.describe()["family"] == "append"
    compare(case, out, lse, label=str(kw))


def test_append_repeat_bitexact():
    case = synth.make_case(name="rep", seed=12, seq_lens=[150, 70], seq_lens_kv=[400, 33],
                           q_heads=32, kv_heads=8, kv_dtype="fp8_e4m3")
    out1, lse1, _, d, _ = run_case(case)
    out2, lse2, _, _, _ = run_case(case, d=d)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)
