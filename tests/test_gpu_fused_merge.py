"""The decode kernel's opt-in in-kernel merge of split rows (the CTA that writes a row
group's last chunk merges it): parity with the oracle, bit-identity with the
separate merge kernel where both modes run the same attention kernel, counters
that reset themselves between launches, and a bounded failure path.

The in-kernel merge lives in the tensor-memory decode kernel; without it, tiles
of at most 16 packed rows run the warp-per-item kernel instead, so for those
cases the two modes agree with the oracle but not bit for bit."""
import numpy as np
import pytest
import torch

import synth
from synth.device import to_device
from gpu_helpers import num_sms, run_case, compare

pytestmark = pytest.mark.gpu

CASES = [
    dict(seq_lens=[1, 1, 1], seq_lens_kv=[3000, 513, 64], q_heads=32, kv_heads=8, chunk_size=512),
    dict(seq_lens=[6, 6, 3], seq_lens_kv=[2500, 1030, 5000], q_heads=64, kv_heads=8,
         chunk_size=1024),
    dict(seq_lens=[2, 1], seq_lens_kv=[700, 129], q_heads=16, kv_heads=2, chunk_size=128,
         kv_dtype="fp8_e4m3", scale_kind="per_kv_head"),
    dict(seq_lens=[1], seq_lens_kv=[40000], q_heads=8, kv_heads=1, chunk_size=256),  # 157 chunks
]


def _run(case, fused):
    import paged_quantized_kv_gqa_gb300 as pa
    pa.pa_set_fused_merge(fused)
    try:
        out, lse, plan, d, st = run_case(case)
    finally:
        pa.pa_set_fused_merge(False)
    assert plan.describe()["fused_merge"] == fused
    return out, lse


@pytest.mark.parametrize("kw", CASES)
def test_fused_merge_matches_oracle_and_separate_merge(kw):
    case = synth.make_case(name="fm", seed=41, **kw)
    of, lf = _run(case, True)
    compare(case, of, lf, label=f"fused merge {kw}")
    os_, ls = _run(case, False)
    compare(case, os_, ls, label=f"separate merge {kw}")
    rows = max(kw["seq_lens"]) * kw["q_heads"] // kw["kv_heads"]
    if rows > 16:   # both modes run the tensor-memory kernel
        assert np.array_equal(of.view(np.uint32), os_.view(np.uint32))
        assert np.array_equal(lf.view(np.uint32), ls.view(np.uint32))


def test_fused_merge_counters_reset_between_launches():
    """One upload, several launches: each launch merges every row again."""
    import paged_quantized_kv_gqa_gb300 as pa
    case = synth.make_case(name="fm-rep", seed=42, seq_lens=[1, 6, 2], seq_lens_kv=[1500, 900, 2100],
                           q_heads=32, kv_heads=8, chunk_size=256)
    d = to_device(case)
    pa.pa_set_fused_merge(True)
    try:
        plan = pa.pa_plan(pa.problem_of(case), case.seq_lens, case.seq_lens_kv,
                          case.cu_seqlens_q, num_sms())
    finally:
        pa.pa_set_fused_merge(False)
    assert plan.describe()["fused_merge"]
    ws = torch.zeros(plan.workspace_size, dtype=torch.uint8, device="cuda")
    args = pa.make_args(q=d["q"], cache_k=d["cache_k"], cache_v=d["cache_v"],
                        k_scale=d["k_scale"], v_scale=d["v_scale"], block_table=d["block_table"],
                        out=d["out"], lse=d["lse"])
    pa.pa_plan_upload(plan, ws)
    first = None
    for _ in range(3):
        d["out"].zero_()
        d["lse"].zero_()
        pa.pa_run(plan, args, ws)
        pa.pa_merge(plan, args, ws)   # a no-op for this plan
        st, det = pa.pa_check(plan, ws)
        assert st == 0, (st, det)
        o = d["out"].float().cpu().numpy()
        l = d["lse"].cpu().numpy()
        if first is None:
            first = (o, l)
            compare(case, o, l, label="fused merge, first launch")
        else:
            assert np.array_equal(o.view(np.uint32), first[0].view(np.uint32))
            assert np.array_equal(l.view(np.uint32), first[1].view(np.uint32))


def test_fused_merge_failure_is_bounded():
    """A loader that skips its first page load: the merge warps' wait ends with
    the rest of the CTA (PA_ERR_DEVICE_TIMEOUT), and a fresh plan runs right."""
    import paged_quantized_kv_gqa_gb300 as pa
    case = synth.make_case(name="fm-to", seed=43, seq_lens=[1], seq_lens_kv=[600], q_heads=8,
                           kv_heads=2, chunk_size=128)
    d = to_device(case)
    pa.pa_debug_set_faults(wait_limit_ns=200_000_000, skip_first_load=True)
    pa.pa_set_fused_merge(True)
    try:
        _, _, plan, _, st = run_case(case, d, sms=1, check=False)
    finally:
        pa.pa_debug_set_faults(0, False)
        pa.pa_set_fused_merge(False)
    assert plan.describe()["fused_merge"]
    assert st == pa.PA_ERR_DEVICE_TIMEOUT
    out, lse, _, _, st2 = run_case(case, d)
    assert st2 == 0
    compare(case, out, lse, label="fused merge after timeout")
