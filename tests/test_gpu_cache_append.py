"""GPU parity of the cache-append step (quantise-and-write of the appended
tokens' K / V into the paged cache) against the oracle: every cache byte must
match exactly."""
import numpy as np
import pytest
import torch

import synth
from synth.cases import new_kv
from synth.device import to_device
from oracle import cache_append as ca
from oracle import attention as oa
from gpu_helpers import num_sms, compare

pytestmark = pytest.mark.gpu


def _append_on_gpu(case, packed=False, misaligned=False):
    import paged_quantized_kv_gqa_gb300 as pa
    d = to_device(case, generate_on_device=False)
    k, v = new_kv(case)
    T = case.total_q
    if case.layout == "mla":
        k_dev = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).cuda()
        v_dev, stride = None, case.head_dim_qk
    elif packed:
        # K and V rows inside a packed qkv tensor [T, (Hq + 2 Hkv) * D]
        D, Hq, Hkv = case.head_dim_qk, case.q_heads, case.kv_heads
        qkv = torch.zeros((T, (Hq + 2 * Hkv) * D), dtype=torch.bfloat16, device="cuda")
        qkv[:, Hq * D:(Hq + Hkv) * D] = torch.from_numpy(
            k.reshape(T, -1).view(np.int16)).view(torch.bfloat16).cuda()
        qkv[:, (Hq + Hkv) * D:] = torch.from_numpy(
            v.reshape(T, -1).view(np.int16)).view(torch.bfloat16).cuda()
        k_dev, v_dev, stride = qkv[:, Hq * D:], qkv[:, (Hq + Hkv) * D:], (Hq + 2 * Hkv) * D
    elif misaligned:
        # rows that start 2 bytes past a 16-byte boundary: the kernel's 2-byte path
        stride = case.kv_heads * case.head_dim_qk + 1
        kb = torch.zeros(T * stride + 1, dtype=torch.bfloat16, device="cuda")
        vb = torch.zeros(T * stride + 1, dtype=torch.bfloat16, device="cuda")
        k_dev = kb[1:].view(T, stride)
        v_dev = vb[1:].view(T, stride)
        k_dev[:, :stride - 1] = torch.from_numpy(k.reshape(T, -1).view(np.int16)).view(torch.bfloat16).cuda()
        v_dev[:, :stride - 1] = torch.from_numpy(v.reshape(T, -1).view(np.int16)).view(torch.bfloat16).cuda()
    else:
        k_dev = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).cuda()
        v_dev = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda()
        stride = case.kv_heads * case.head_dim_qk
    plan = pa.pa_plan(pa.problem_of(case), case.seq_lens, case.seq_lens_kv, case.cu_seqlens_q,
                      num_sms())
    ws = torch.zeros(max(plan.workspace_size, 256), dtype=torch.uint8, device="cuda")
    args = pa.make_args(q=d["q"], cache_k=d["cache_k"], cache_v=d["cache_v"],
                        k_scale=d["k_scale"], v_scale=d["v_scale"], block_table=d["block_table"],
                        out=d["out"], lse=d["lse"], seq_lens=d["seq_lens"],
                        seq_lens_kv=d["seq_lens_kv"], cu_seqlens_q=d["cu_seqlens_q"])
    pa.pa_plan_upload(plan, ws)
    pa.pa_cache_append(plan, args, k_dev, v_dev, stride, ws)
    st, det = pa.pa_check(plan, ws)
    assert st == 0, (st, det, pa.pa_last_error())
    ck = d["cache_k"].cpu().numpy()
    cv = None if case.layout == "mla" else d["cache_v"].cpu().numpy()
    ref_k, ref_v = ca.cache_append(case, k, v, case.cache_k,
                                   None if case.layout == "mla" else case.cache_v)
    return ck, cv, ref_k, ref_v, d, plan, ws, args


CASES = [
    dict(seq_lens=[70, 3, 0, 130], seq_lens_kv=[100, 0, 9, 63], q_heads=32, kv_heads=8),
    dict(seq_lens=[40, 65], seq_lens_kv=[64, 1], q_heads=16, kv_heads=4, scale_kind="per_channel"),
    dict(seq_lens=[90, 1], seq_lens_kv=[500, 127], q_heads=32, kv_heads=8, kv_dtype="fp8_e4m3"),
    dict(seq_lens=[33], seq_lens_kv=[31], q_heads=8, kv_heads=2, scale_kind="global"),
]


@pytest.mark.parametrize("kw", CASES)
def test_cache_append_bitexact(kw):
    case = synth.make_case(name="append-cache", seed=17, **kw)
    ck, cv, rk, rv, *_ = _append_on_gpu(case)
    assert np.array_equal(ck, rk), f"K bytes differ at {np.argwhere(ck != rk)[:4]}"
    assert np.array_equal(cv, rv), f"V bytes differ at {np.argwhere(cv != rv)[:4]}"


def test_cache_append_from_packed_qkv():
    case = synth.make_case(name="append-qkv", seed=18, seq_lens=[50, 20], seq_lens_kv=[10, 200],
                           q_heads=16, kv_heads=4)
    ck, cv, rk, rv, *_ = _append_on_gpu(case, packed=True)
    assert np.array_equal(ck, rk) and np.array_equal(cv, rv)


def test_cache_append_misaligned_rows():
    """New rows that are only 2-byte aligned take the kernel's 2-byte path."""
    case = synth.make_case(name="append-mis", seed=20, seq_lens=[45, 70], seq_lens_kv=[19, 128],
                           q_heads=16, kv_heads=4, scale_kind="per_channel")
    ck, cv, rk, rv, *_ = _append_on_gpu(case, misaligned=True)
    assert np.array_equal(ck, rk) and np.array_equal(cv, rv)


def test_cache_append_mla_rows():
    case = synth.make_case(name="append-mla", seed=19, seq_lens=[2, 1, 2], seq_lens_kv=[63, 64, 300],
                           q_heads=128, kv_heads=1, head_dim_qk=576, head_dim_v=512,
                           layout="mla", kv_dtype="fp8_e4m3", scale_kind="global",
                           sm_scale=1.0 / np.sqrt(192.0))
    ck, _, rk, _, *_ = _append_on_gpu(case)
    assert np.array_equal(ck, rk)


def test_append_workload_cache_then_attention():
    """The append workload's new tokens quantised into the cache by the kernel,
    then attention over the updated cache against the oracle."""
    import paged_quantized_kv_gqa_gb300 as pa
    case = synth.config(3)
    ck, cv, rk, rv, d, plan, ws, args = _append_on_gpu(case)
    assert np.array_equal(ck, rk) and np.array_equal(cv, rv)
    pa.pa_run(plan, args, ws)
    pa.pa_merge(plan, args, ws)
    st, det = pa.pa_check(plan, ws)
    assert st == 0, (st, det)
    case._cache_k, case._cache_v, case._page_memo = rk, rv, {}
    out = d["out"].float().cpu().numpy()
    lse = d["lse"].cpu().numpy()
    units = [(b, (5 * b + 2) % case.kv_heads) for b in range(case.bsz)]
    compare(case, out, lse, units=units, label="append-3 after cache append")
