"""pa_run_static: the attention path with the library's built-in workspace.

Callers such as plugins whose host framework owns all device allocations, or
real-time loops that must not allocate, cannot hand the library a workspace
from cudaMalloc; pa_run_static serves them from a fixed 32 MiB static device
buffer.  These checks call it through the C ABI and compare its output with
the ordinary entry points (caller workspace) and with the fp64 oracle on two
calls in a row, and check that a call's device status starts clean.  The file
is named to be collected last, so a stop-at-first-failure run has already run
every other test.
"""
import numpy as np
import pytest
import torch

import synth
from synth.device import to_device
from gpu_helpers import run_case, compare, OUT_ATOL, OUT_RTOL, LSE_ATOL, num_sms

pytestmark = pytest.mark.gpu


def _args(pa, d, out, lse):
    return pa.make_args(q=d["q"], cache_k=d["cache_k"], cache_v=d["cache_v"],
                        k_scale=d["k_scale"], v_scale=d["v_scale"],
                        block_table=d["block_table"], out=out, lse=lse)


def test_static_workspace_matches_caller_workspace_twice():
    import paged_quantized_kv_gqa_gb300 as pa
    case = synth.make_case(name="static", seed=21, seq_lens=[1, 3, 2, 1],
                           seq_lens_kv=[1500, 700, 2049, 64], q_heads=32, kv_heads=8,
                           scale_kind="per_channel", chunk_size=512)
    d = to_device(case)
    ref_out, ref_lse, plan, _, _ = run_case(case, d)      # existing entry points
    assert plan.describe()["max_chunks"] > 1               # the partial states are used
    for _ in range(2):
        out = torch.full_like(d["out"], float("nan"))
        lse = torch.full_like(d["lse"], float("nan"))
        pa.pa_run_static(plan, _args(pa, d, out, lse), check=True)
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        assert np.all(np.abs(o - ref_out) <= OUT_ATOL + OUT_RTOL * np.abs(ref_out))
        assert np.all(np.abs(l - ref_lse) <= LSE_ATOL)
        compare(case, o, l, label="static workspace")          # against the oracle as well


def test_static_workspace_status_is_cleared_between_calls():
    """A call that meets a block-table entry outside the pool reports it; the
    next clean call on the same built-in buffer reports success."""
    import paged_quantized_kv_gqa_gb300 as pa
    case = synth.make_case(name="static-bad", seed=23, seq_lens=[1, 1], seq_lens_kv=[300, 90],
                           q_heads=8, kv_heads=2, chunk_size=128)
    d = to_device(case)
    plan = pa.pa_plan(pa.problem_of(case), case.seq_lens, case.seq_lens_kv,
                      case.cu_seqlens_q, num_sms())
    good = d["block_table"].clone()
    d["block_table"][0, 1] = case.num_pages + 7
    out = torch.zeros_like(d["out"])
    lse = torch.zeros_like(d["lse"])
    with pytest.raises(pa.PaError) as e:
        pa.pa_run_static(plan, _args(pa, d, out, lse), check=True)
    assert e.value.status == pa.PA_ERR_BAD_PAGE
    d["block_table"].copy_(good)
    pa.pa_run_static(plan, _args(pa, d, out, lse), check=True)
    compare(case, out.float().cpu().numpy(), lse.cpu().numpy(), label="static after a bad page")


def test_static_workspace_rejects_oversized_plans():
    import paged_quantized_kv_gqa_gb300 as pa
    case = synth.make_case(name="big", seed=22, seq_lens=[6] * 64,
                           seq_lens_kv=[30000] * 64, q_heads=64, kv_heads=8, chunk_size=1024)
    plan = pa.pa_plan(pa.problem_of(case), case.seq_lens, case.seq_lens_kv,
                      case.cu_seqlens_q, num_sms())
    assert plan.workspace_size > 32 << 20
    null = pa.make_args(q=16, cache_k=16, cache_v=16, k_scale=16, v_scale=16,
                        block_table=16, out=16)
    with pytest.raises(pa.PaError) as e:
        pa.pa_run_static(plan, null)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    assert "built-in buffer" in pa.pa_last_error()
