"""Shared helpers for the GPU parity tests: run a synthetic case through the C
ABI and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import synth
from synth.device import to_device
from oracle import attention as oa

OUT_ATOL = 1e-2
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3


def num_sms() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def run_case(case, d=None, sms=None, check=True):
    """Plan, upload, run and merge one case on cuda:0; returns (out, lse, plan, tensors)."""
    import paged_quantized_kv_gqa_gb300 as pa
    if d is None:
        d = to_device(case)
    plan = pa.pa_plan(pa.problem_of(case), case.seq_lens, case.seq_lens_kv, case.cu_seqlens_q,
                      sms or num_sms())
    ws = torch.zeros(max(plan.workspace_size, 256), dtype=torch.uint8, device="cuda")
    args = pa.make_args(q=d["q"], cache_k=d["cache_k"], cache_v=d["cache_v"],
                        k_scale=d["k_scale"], v_scale=d["v_scale"], block_table=d["block_table"],
                        out=d["out"], lse=d["lse"], seq_lens=d["seq_lens"],
                        seq_lens_kv=d["seq_lens_kv"], cu_seqlens_q=d["cu_seqlens_q"],
                        attn_mask=d.get("attn_mask"))
    pa.pa_plan_upload(plan, ws)
    pa.pa_run(plan, args, ws)
    pa.pa_merge(plan, args, ws)
    st, det = pa.pa_check(plan, ws)
    if check:
        assert st == 0, f"device status {st} detail {det}: {pa.pa_last_error()}"
    out = d["out"].float().cpu().numpy()
    lse = d["lse"].cpu().numpy()
    return out, lse, plan, d, st


def _ref_worker(cfg, units):
    import synth as _s
    from oracle import attention as _oa
    return _oa.reference(_s.config(cfg), units)


def reference_all(cfg: int, case):
    """The oracle over every (sequence, kv head) unit of named workload cfg, the
    units shared out over the host cores (spawned processes that rebuild the
    workload: a process forked after CUDA initialisation would hang)."""
    import multiprocessing as mp
    import os
    units = [(b, h) for b in range(case.bsz) for h in range(case.kv_heads) if case.seq_lens[b] > 0]
    n = max(1, min(len(units), os.cpu_count() or 1))
    parts = [units[i::n] for i in range(n)]
    with mp.get_context("spawn").Pool(n) as pool:
        got = pool.starmap(_ref_worker, [(cfg, u) for u in parts])
    ref_o, ref_l = got[0]
    for o, l in got[1:]:
        rows = ~np.isnan(l)
        ref_o[rows] = o[rows]
        ref_l[rows] = l[rows]
    return ref_o, ref_l


def compare(case, out, lse, units=None, label="", ref=None):
    """Element-wise check against the oracle on the given (b, kv head) units
    (or against a precomputed oracle result `ref`)."""
    ref_o, ref_l = ref if ref is not None else oa.reference(case, units)
    rows = ~np.isnan(ref_l)
    assert rows.any(), "nothing compared"
    o = out[rows]
    r = ref_o[rows]
    # a NaN would compare false against the tolerance below
    assert np.isfinite(o).all(), f"{label}: {int((~np.isfinite(o)).sum())} non-finite output elements"
    err = np.abs(o - r)
    tol = OUT_ATOL + OUT_RTOL * np.abs(r)
    bad = err > tol
    rms = float(np.sqrt(np.mean(r * r))) or 1.0
    msg = (f"{label}: out max err {err.max():.3e} (max err / rms {err.max() / rms:.3e}), "
           f"{int(bad.sum())} of {bad.size} outside 1e-2 + 1e-2|ref|")
    assert not bad.any(), msg
    dl = np.abs(lse[rows] - ref_l[rows])
    both_inf = np.isneginf(lse[rows]) & np.isneginf(ref_l[rows])
    dl[both_inf] = 0.0
    assert dl.max() <= LSE_ATOL, f"{label}: lse max err {dl.max():.3e}"
    # diagnostic: how much of the tolerance the worst element uses
    print(f"{label}: max |err| / tol = {float((err / tol).max()):.3f} (out), "
          f"{float(dl.max()) / LSE_ATOL:.3f} (lse); {bad.size} elements")
    return float(err.max()), float(dl.max())
