"""GPU parity of speculative verify with a draft-tree mask (the decode family
with attn_mask) against the fp64 oracle."""
import numpy as np
import pytest

import synth
from synth.cases import tree_mask
from gpu_helpers import run_case, compare

pytestmark = pytest.mark.gpu

EDGE = [
    dict(seq_lens=[6, 6, 3], seq_lens_kv=[500, 64, 1000], q_heads=64, kv_heads=8, chunk_size=128),
    dict(seq_lens=[6, 2], seq_lens_kv=[0, 130], q_heads=64, kv_heads=8, chunk_size=0),
    dict(seq_lens=[8, 5, 1], seq_lens_kv=[200, 7, 63], q_heads=32, kv_heads=4, chunk_size=64,
         kv_dtype="fp8_e4m3"),
    dict(seq_lens=[16], seq_lens_kv=[300], q_heads=8, kv_heads=2, scale_kind="per_channel",
         chunk_size=256),
]


@pytest.mark.parametrize("kw", EDGE)
def test_tree_mask_decode_edge_cases(kw):
    case = synth.make_case(name="tree", seed=23, **kw)
    case.attn_mask = tree_mask(case)
    out, lse, plan, _, _ = run_case(case)
    assert plan.describe()["family"] == "decode"
    compare(case, out, lse, label="tree " + str(kw))


def test_spec_verify_4_tree_mask_sampled():
    """Full-size speculative-verify workload with a seeded draft tree per sequence."""
    case = synth.config(4)
    case.attn_mask = tree_mask(case)
    out, lse, plan, _, _ = run_case(case)
    rng = np.random.default_rng(1)
    bs = sorted(set(rng.choice(case.bsz, 8, replace=False).tolist()) | {case.bsz - 1})
    compare(case, out, lse, units=[(b, int(rng.integers(case.kv_heads))) for b in bs],
            label="spec-verify-4 tree")


def test_tree_mask_rejected_outside_decode_family():
    import paged_quantized_kv_gqa_gb300 as pa
    case = synth.make_case(name="tree-append", seed=24, seq_lens=[40], seq_lens_kv=[10],
                           q_heads=32, kv_heads=8)
    case.attn_mask = tree_mask(case)
    with pytest.raises(pa.PaError) as e:
        run_case(case)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
