"""GPU parity of the fused output epilogue (shift_bias, smooth_weight, bf16 or
int8 output) against the oracle, for one-chunk rows (written by the attention
kernels) and split rows (written by the merge)."""
import numpy as np
import pytest
import torch

import synth
from synth.device import to_device
from synth.formats import to_bf16_bits
from oracle import attention as oa
from oracle import epilogue as ep
from gpu_helpers import num_sms, OUT_ATOL, OUT_RTOL, LSE_ATOL

pytestmark = pytest.mark.gpu


def _run(case, int8_out, in_scale=0.5):
    import paged_quantized_kv_gqa_gb300 as pa
    d = to_device(case)
    HqDv = case.q_heads * case.head_dim_v
    r = np.random.default_rng(case.seed)
    shift = to_bf16_bits(r.normal(0.0, 0.1, HqDv).astype(np.float32))
    smooth = to_bf16_bits(r.uniform(0.5, 1.5, HqDv).astype(np.float32))
    sh = torch.from_numpy(shift.view(np.int16)).view(torch.bfloat16).cuda()
    sm = torch.from_numpy(smooth.view(np.int16)).view(torch.bfloat16).cuda()
    T = case.total_q
    out = (torch.zeros((T, case.q_heads, case.head_dim_v), dtype=torch.int8, device="cuda")
           if int8_out else d["out"])
    plan = pa.pa_plan(pa.problem_of(case), case.seq_lens, case.seq_lens_kv, case.cu_seqlens_q,
                      num_sms())
    ws = torch.zeros(max(plan.workspace_size, 256), dtype=torch.uint8, device="cuda")
    args = pa.make_args(q=d["q"], cache_k=d["cache_k"], cache_v=d["cache_v"],
                        k_scale=d["k_scale"], v_scale=d["v_scale"], block_table=d["block_table"],
                        out=out, lse=d["lse"], seq_lens=d["seq_lens"],
                        seq_lens_kv=d["seq_lens_kv"], cu_seqlens_q=d["cu_seqlens_q"],
                        shift_bias=sh, smooth_weight=sm, out_int8=int8_out, in_scale=in_scale,
                        quant_max_bound=127.0, quant_min_bound=-127.0)
    pa.pa_plan_upload(plan, ws)
    pa.pa_run(plan, args, ws)
    pa.pa_merge(plan, args, ws)
    st, det = pa.pa_check(plan, ws)
    assert st == 0, (st, det, pa.pa_last_error())
    ref_o, ref_l = oa.reference(case)
    ref = ep.apply(ref_o, shift, smooth)
    rows = ~np.isnan(ref_l)
    lse = d["lse"].cpu().numpy()
    dl = np.abs(lse[rows] - ref_l[rows])
    dl[np.isneginf(lse[rows]) & np.isneginf(ref_l[rows])] = 0
    assert dl.max() <= LSE_ATOL
    if int8_out:
        got = out.cpu().numpy().astype(np.int64)[rows]
        want = ep.quantize_int8(ref, in_scale, 127.0, -127.0)[rows]
        slack = np.ceil(127.0 * in_scale * (OUT_ATOL + OUT_RTOL * np.abs(ref[rows]))) + 1
        bad = np.abs(got - want) > slack
        assert not bad.any(), f"{int(bad.sum())} int8 codes off by more than the tolerance"
        # not a degenerate quantisation, and no systematic offset between the codes
        assert (got != 0).any() and np.ptp(want) > 10
        assert np.mean(np.abs(got - want)) <= 1.0
    else:
        got = out.float().cpu().numpy()[rows]
        err = np.abs(got - ref[rows])
        assert (err <= OUT_ATOL + OUT_RTOL * np.abs(ref[rows])).all(), err.max()
    return plan.describe()


CASES = [
    ("decode", dict(seq_lens=[1, 1, 6], seq_lens_kv=[40, 700, 300], q_heads=32, kv_heads=8,
                    chunk_size=256)),
    # one token per sequence, group of 4: the decode kernel's epilogue warpgroup writes the rows
    ("decode", dict(seq_lens=[1, 1, 1], seq_lens_kv=[40, 700, 300], q_heads=32, kv_heads=8,
                    chunk_size=256)),
    ("append", dict(seq_lens=[70, 130], seq_lens_kv=[30, 600], q_heads=32, kv_heads=8,
                    chunk_size=256)),
    ("append", dict(seq_lens=[90], seq_lens_kv=[100], q_heads=16, kv_heads=4,
                    kv_dtype="fp8_e4m3")),
    ("mla", dict(seq_lens=[2, 1], seq_lens_kv=[500, 64], q_heads=128, kv_heads=1,
                 head_dim_qk=576, head_dim_v=512, layout="mla", kv_dtype="fp8_e4m3",
                 scale_kind="global", chunk_size=128, sm_scale=1.0 / np.sqrt(192.0))),
]


@pytest.mark.parametrize("int8_out", [False, True])
@pytest.mark.parametrize("family,kw", CASES)
def test_output_epilogue(family, kw, int8_out):
    case = synth.make_case(name="epi", seed=31, **kw)
    desc = _run(case, int8_out)
    assert desc["family"] == family
