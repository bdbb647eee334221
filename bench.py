"""Benchmark of the paged, quantised-KV attention path on one GB300.

One step = the whole path over one batch: pa_run (attention over the paged
int8 / FP8 cache, split-KV partials) + pa_merge (log-sum-exp merge), with the
plan already uploaded and every input resident in HBM.

By default every named workload runs, one after the other, and the single JSON
line carries them all:
  * the headline is decode-2 (bsz 64, q_len 1, 32 q heads / 8 kv heads, head
    dim 128, int8 per-channel scales, prefix U[512, 4096], 4096-page shuffled
    pool, chunk 512): its metric is algorithmic KV-cache bytes per second, the
    bytes of every visible position's K and V rows read once (per token, not
    rounded up to pages);
  * config.per_workload holds one record per workload: decode-1 (latency in
    microseconds: a two-sequence step is launch-bound), decode-2 and
    spec-verify-4 (GB/s against the HBM copy peak), append-3 and mla-5
    (algorithmic FLOP/s, 2 (Dqk + Dv) per visible (query head, position) pair,
    against the tensor peak), each with its own roofline, end-to-end figure,
    clock record and oracle CPU baseline.
--config N runs one workload only (its record is then the headline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl reference]

For N > 1 it runs under torch.distributed (one process per GPU); each rank runs
an independent replica of the workload (the path has no cross-GPU exchange),
time = max over ranks, value = all ranks' work / time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "KV-cache HBM GB/s (decode) & TFLOP/s (append/MLA), % of GB300 roofline"
L2_BYTES = 129 * 1000 * 1000          # GB300 L2 (129 MB)
L2_FLUSH_BYTES = 512 << 20
L2_DRAIN_BYTES = 256 << 20
L2_NOTE = ("flushed before every timed step: 512 MiB written, then 256 MiB read so that the "
           "flush's dirty lines are written back before the timed region, not during it")
ROT_MAX = 8                           # most cache copies a step rotation may use


def rotation(kv_bytes: int) -> int:
    """Cache copies the timed steps rotate over: at least two (a step never
    reads the copy the previous step read), and enough that more than twice
    the L2 size is read between two uses of one copy; 0 when that would take
    more than ROT_MAX copies (such a small workload is timed with a flush)."""
    n = max(2, 1 + -(-2 * L2_BYTES // max(1, kv_bytes)))
    return n if n <= ROT_MAX else 0


def rotation_note(n_rot: int, kv_bytes: int) -> str:
    if n_rot == 0:
        return L2_NOTE
    return (f"not flushed: inputs larger than L2; steps rotate over {n_rot} copies of the cache "
            f"({kv_bytes / 1e6:.0f} MB read per step, so {(n_rot - 1) * kv_bytes / 1e6:.0f} MB "
            f"> 2x L2 is read between two uses of one copy)")


class L2Flush:
    """Evicts the workload from L2 between timed steps: a write of a buffer four
    times the L2 size, then a read of another twice its size, which pushes the
    written (dirty) lines out to HBM before the next timed step starts."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_DRAIN_BYTES // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty(1, dtype=torch.int64, device=dev)

    def __call__(self, i: int):
        self.w.fill_(i & 0xFF)
        self.sink.copy_(self.r.sum().view(1))
HEADLINE = 2
ALL_WORKLOADS = (2, 1, 4, 3, 5)       # headline first


# GB300 nominal peaks, reported beside the measured ones: HBM3e 7.9 TB/s,
# dense bf16 / fp16 tensor 2.25 PFLOP/s
NOMINAL_PEAK = {"hbm": 7900.0, "tensor": 2250.0}


def _peaks(bound: str):
    """(peak, source) for an HBM-bound (GB/s) or tensor-bound (TFLOP/s) kernel.
    The fp16 kind::f16 tensor rate equals the bf16 one the peaks file measures;
    a kernel timed alone takes the burst figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key, fallback = ("hbm_gbs", 6800.0) if bound == "hbm" else ("bf16_tflops", 1900.0)
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if key in d:
            return float(d[key]), f"measured {key}"
    return fallback, f"fallback {key}"


# DRAM bytes (read + written) per launch of each attention kernel, from one
# ncu capture of dram__bytes_read.sum + dram__bytes_write.sum on the workload.
# A figure is reported only while the kernel's sources and the planner (which
# decides the items, hence the partial states written) still hash to the
# version it was taken with.
NCU_TRAFFIC = {
    # decode-2 runs the warp-per-item kernel (at most 16 packed rows)
    "decode-2": (("pa_decode_warp.cu", "pa_index.cuh"), "43caaa15a0fbd4dc", 318.204928e6 + 4.337920e6),
    # captured on the first 16 of the 128 sequences (726.5 MB of the 5443 MB
    # cache) and scaled by the KV-bytes ratio 7.4922: pages read and partial
    # states written both grow per sequence
    "spec-verify-4": (("pa_decode.cu", "pa_index.cuh", "pa_merge.cuh"), "3545fe789aae18a8",
                      (729.481728e6 + 31.898112e6) * 7.492152264116904),
    "append-3": (("pa_append.cu",), "a9cbfbb7a3133fa5", 72.280576e6 + 2.418432e6),
    "mla-5": (("pa_mla.cu",), "bdf0753cd25ebc74", 224.310784e6 + 6.930432e6),
}


def _kernel_sha(files) -> str:
    """Hash of a kernel's source files, the headers every kernel includes and
    the planner."""
    import hashlib
    h = hashlib.sha256()
    for n in tuple(files) + ("pa_common.cuh", "pa_ptx.cuh", "pa_internal.h", "pa_api.cu"):
        with open(os.path.join(ROOT, "paged_quantized_kv_gqa_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(workload: str):
    ent = NCU_TRAFFIC.get(workload)
    if ent is None or ent[1] is None or _kernel_sha(ent[0]) != ent[1]:
        return None
    return int(ent[2])


def _kind(config: int) -> str:
    """latency (decode-1), bytes (HBM-bound decode) or flops (tensor-bound)."""
    return "latency" if config == 1 else "flops" if config in (3, 5) else "bytes"


def algorithmic_bytes(case) -> int:
    """KV bytes every visible position's K and V rows take, read once: per token
    sum_b kvtot_b * Hkv * (Dqk + Dv) bytes (one byte per int8 / e4m3 element);
    MLA reads each 576-byte latent row once (V is its prefix)."""
    kvtot = case.kvtot.astype(np.int64)
    kvtot = kvtot[np.asarray(case.seq_lens) > 0]
    if case.layout == "mla":
        return int(kvtot.sum()) * case.head_dim_qk
    return int(kvtot.sum()) * case.kv_heads * (case.head_dim_qk + case.head_dim_v)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch.distributed as dist
    dist.init_process_group(backend="nccl")
    return dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))


def _max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """Largest per-rank value (the step time the job is charged)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_rate(work_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput of N independent replicas: every rank's work over
    the slowest rank's time (weak scaling)."""
    return work_per_rank * world / (ms_max * 1e-3)


def _barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def _workload(config: int, bsz: int = 0):
    import synth
    return synth.config(config, bsz)


def synth_desc(n: int) -> str:
    import synth
    return synth.CONFIG_NAMES[n]


# ---------------------------------------------------------------- CPU baseline
# The fp64 oracle, as it stands, over (sequence, kv head) units on every host
# core: a process pool forked before any CUDA call (the workers inherit the
# host cases; a pool forked after CUDA initialisation would hang).
_CASES = {}


def _cpu_unit(key, b: int, h: int):
    """One (sequence, kv head) unit of the oracle in a worker: its synthetic cache
    pages are produced first (input generation, untimed), then the oracle runs
    on them.  Returns (work in the metric's unit, seconds of the oracle)."""
    from oracle import attention as oa
    case = _CASES[key]
    case._page_memo = {}
    kvtot = int(case.seq_lens_kv[b]) + int(case.seq_lens[b])
    for lb in range((kvtot + case.block_size - 1) // case.block_size):
        pg = int(case.block_table[b, lb])
        case.page_k(pg)
        if case.layout != "mla":
            case.page_v(pg)
    t0 = time.perf_counter()
    oa.unit_attention(case, b, h)
    return _unit_work(case, b, _kind_of_case(case)), time.perf_counter() - t0


def _kind_of_case(case) -> str:
    return "flops" if case.name.startswith(("append", "mla")) else "bytes"


def _unit_work(case, b: int, kind: str) -> float:
    """Work of one (sequence, kv head) unit in the metric's unit (bytes or flops)."""
    q, pre = float(case.seq_lens[b]), float(case.seq_lens_kv[b])
    if q == 0:
        return 0.0
    if kind == "flops":   # visible (query head, position) pairs x 2 (Dqk + Dv)
        G = case.q_heads // case.kv_heads
        pairs = q * pre + q * (q + 1) / 2 if case.causal else q * (pre + q)
        return pairs * G * 2 * (case.head_dim_qk + case.head_dim_v)
    row = case.head_dim_qk if case.layout == "mla" else case.head_dim_qk + case.head_dim_v
    return (pre + q) * row


class CpuPool:
    """Host cores running the oracle; created before the first GPU call."""

    def __init__(self, cases: dict):
        import multiprocessing as mp
        _CASES.update(cases)
        self.cores = os.cpu_count() or 1
        self.pool = mp.get_context("fork").Pool(self.cores)

    def close(self):
        self.pool.terminate()
        self.pool.join()

    def baseline(self, key, seconds: float) -> dict:
        """The oracle on a bounded sample: batches of one unit per core until
        about `seconds` of oracle CPU time (summed over the cores) are spent;
        the rate is the sample's work over the sum of the batches' wall times."""
        case = _CASES[key]
        kind = _kind_of_case(case)
        units = [(b, h) for b in range(case.bsz) for h in range(case.kv_heads) if case.seq_lens[b] > 0]
        np.random.default_rng(0).shuffle(units)
        cpu_target = max(1.0, seconds)
        done, n, i, wall, cpu = 0.0, 0, 0, 0.0, 0.0
        while i < len(units) and cpu < cpu_target:
            batch = units[i:i + self.cores]
            i += len(batch)
            got = self.pool.starmap(_cpu_unit, [(key, b, h) for b, h in batch])
            done += sum(w for w, _ in got)
            cpu += sum(t for _, t in got)
            wall += max(t for _, t in got)     # the batch's units run side by side
            n += len(batch)
        dt = wall
        scale, unit = (1e12, "TFLOP/s") if kind == "flops" else (1e9, "GB/s")
        return {"value": round(done / dt / scale, 6), "unit": unit, "cores": self.cores,
                "kind": "oracle",
                "sample": f"{n} of {len(units)} (sequence, kv head) units of {case.name} in batches "
                          f"of one unit per core: {cpu:.1f} s of oracle CPU time, {dt:.2f} s wall "
                          f"(slowest unit of each batch) on {self.cores} processes, numpy fp64; the "
                          f"synthetic cache pages are generated before each unit, untimed"}


# ---------------------------------------------------------------- GPU workload
def run_workload(cfg: int, case, args, world: int, local: int, dev, pool) -> dict:
    """Times one workload; returns its record (the fields of the JSON line)."""
    import torch
    import paged_quantized_kv_gqa_gb300 as pa
    from synth.device import to_device

    kind = _kind(cfg)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    d = to_device(case, dev)
    if args.fused_merge:
        pa.pa_set_fused_merge(True)
    plan = pa.pa_plan(pa.problem_of(case), case.seq_lens, case.seq_lens_kv, case.cu_seqlens_q, sms)
    pa.pa_set_fused_merge(False)
    desc = plan.describe()
    ws = torch.zeros(plan.workspace_size, dtype=torch.uint8, device=dev)
    cargs = pa.make_args(q=d["q"], cache_k=d["cache_k"], cache_v=d["cache_v"],
                         k_scale=d["k_scale"], v_scale=d["v_scale"], block_table=d["block_table"],
                         out=d["out"], lse=d["lse"], seq_lens=d["seq_lens"],
                         seq_lens_kv=d["seq_lens_kv"], cu_seqlens_q=d["cu_seqlens_q"],
                         attn_mask=d.get("attn_mask"))
    stream = torch.cuda.current_stream(dev)
    pa.pa_plan_upload(plan, ws, stream)
    flush = L2Flush(dev)
    split = desc["max_chunks"] > 1 and not desc["fused_merge"]
    kv_bytes = algorithmic_bytes(case)

    # the cache is not in L2 when a step starts: the steps rotate over copies
    # of it (inputs larger than L2), or, for a workload too small for that,
    # L2 is flushed before every step
    n_rot = rotation(kv_bytes)
    same_kv = d["cache_v"].data_ptr() == d["cache_k"].data_ptr()
    caches = [(d["cache_k"], d["cache_v"])]
    for _ in range(n_rot - 1):
        ck = d["cache_k"].clone()
        caches.append((ck, ck if same_kv else d["cache_v"].clone()))

    def args_for(ck, cv, q, bt, out, lse):
        return pa.make_args(q=q, cache_k=ck, cache_v=cv, k_scale=d["k_scale"],
                            v_scale=d["v_scale"], block_table=bt, out=out, lse=lse,
                            seq_lens=d["seq_lens"], seq_lens_kv=d["seq_lens_kv"],
                            cu_seqlens_q=d["cu_seqlens_q"], attn_mask=d.get("attn_mask"))
    rargs = [args_for(ck, cv, d["q"], d["block_table"], d["out"], d["lse"]) for ck, cv in caches]

    def timed(K: int, flushed: bool, mid: bool):
        """K steps; events around each step and, with mid, also between the
        attention kernel and the merge (an event there keeps the merge, a
        programmatic dependent launch, from being set up during the attention
        kernel's last CTAs, so steps are timed without it)."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            if flushed:
                flush(i)                       # evict the cache from L2 between steps
            a, m, b = ev[i]
            ak = cargs if flushed else rargs[i % len(rargs)]
            a.record(stream)
            pa.pa_run(plan, ak, ws, stream)
            if mid:
                m.record(stream)
            if split:
                pa.pa_merge(plan, ak, ws, stream)
            b.record(stream)
        return ev

    for i in range(max(args.warmup, len(rargs))):
        if n_rot == 0:
            flush(1)
        ak = rargs[i % len(rargs)]
        pa.pa_run(plan, ak, ws, stream)
        if split:
            pa.pa_merge(plan, ak, ws, stream)
    st, det = pa.pa_check(plan, ws, stream)
    if st != 0:
        raise RuntimeError(f"{case.name}: device status {st} ({pa.pa_last_error()})")

    K = args.steps
    _barrier(world)
    torch.cuda.synchronize(dev)
    with Clocks(local) as clk:
        ev = timed(K, n_rot == 0, mid=False)   # the steps
        evk = timed(K, n_rot == 0, mid=True)   # the same steps, the attention kernel timed alone
        torch.cuda.synchronize(dev)
    _barrier(world)
    step_ms = [a.elapsed_time(b) for a, _, b in ev]
    run_ms = [a.elapsed_time(m) for a, m, _ in evk]
    ms = statistics.mean(step_ms)
    ms_max = _max_over_ranks(ms, world)
    run_mean = statistics.mean(run_ms)
    st, det = pa.pa_check(plan, ws, stream)
    if st != 0:
        raise RuntimeError(f"{case.name}: device status {st} ({pa.pa_last_error()})")
    # the same steps with L2 flushed before each (reported beside the number)
    flushed_ms = None
    if n_rot:
        evf = timed(K, True, mid=False)
        torch.cuda.synchronize(dev)
        flushed_ms = _max_over_ranks(statistics.mean(a.elapsed_time(b) for a, _, b in evf), world)
    if kind == "flops":
        work, unit, bound = desc["flops"] / 1e12, "TFLOP/s", "tensor"
    else:
        work, unit, bound = kv_bytes / 1e9, "GB/s", "hbm"
    peak, peak_kind = _peaks(bound)
    achieved = work / (run_mean * 1e-3)
    launches = K * (2 if split else 1)

    # end to end through the public API with host buffers, as a serving loop
    # runs it: every step uploads its inputs (q, block table, plan) from pinned
    # host memory, runs, merges and reads its output and lse back into pinned
    # host memory.  Two sets of device inputs / outputs / workspaces alternate,
    # so step i+1's upload (copy stream) and step i-1's download (second copy
    # stream) overlap step i's kernels; events order each buffer's reuse.  The
    # timed region runs from the first upload to the last result in host
    # memory.  L2 is not flushed in between; the steps rotate over the same
    # cache copies as the kernel-timed steps (a flush-timed workload, too small
    # for a rotation, uses its one cache here).
    q_h = d["q"].cpu().pin_memory()
    bt_h = d["block_table"].cpu().pin_memory()
    h2d = q_h.numel() * q_h.element_size() + bt_h.numel() * 4 + desc["plan_bytes"]
    d2h = d["out"].numel() * d["out"].element_size() + d["lse"].numel() * 4
    sets = []
    for k in range(2):
        qk = torch.empty_like(d["q"])
        btk = torch.empty_like(d["block_table"])
        outk = torch.empty_like(d["out"])
        lsek = torch.empty_like(d["lse"])
        wsk = torch.zeros(plan.workspace_size, dtype=torch.uint8, device=dev)
        ak = [args_for(ck, cv, qk, btk, outk, lsek) for ck, cv in caches]
        sets.append(dict(q=qk, bt=btk, out=outk, lse=lsek, ws=wsk, args=ak,
                         out_h=torch.empty_like(d["out"], device="cpu").pin_memory(),
                         lse_h=torch.empty_like(d["lse"], device="cpu").pin_memory()))
    up_s, down_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n_e2e = max(8, K)

    def e2e_pass():
        ev_up = [torch.cuda.Event() for _ in range(n_e2e)]
        ev_run = [torch.cuda.Event() for _ in range(n_e2e)]
        ev_down = [torch.cuda.Event() for _ in range(n_e2e)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        t0.record(up_s)
        for i in range(n_e2e):
            sk = sets[i & 1]
            if i >= 2:
                up_s.wait_event(ev_run[i - 2])      # step i-2 has read this set's inputs
            with torch.cuda.stream(up_s):
                sk["q"].copy_(q_h, non_blocking=True)
                sk["bt"].copy_(bt_h, non_blocking=True)
            pa.pa_plan_upload(plan, sk["ws"], up_s)
            ev_up[i].record(up_s)
            stream.wait_event(ev_up[i])
            if i >= 2:
                stream.wait_event(ev_down[i - 2])   # step i-2's result has left this set's out
            ak = sk["args"][i % len(caches)]
            pa.pa_run(plan, ak, sk["ws"], stream)
            if split:
                pa.pa_merge(plan, ak, sk["ws"], stream)
            ev_run[i].record(stream)
            down_s.wait_event(ev_run[i])
            with torch.cuda.stream(down_s):
                sk["out_h"].copy_(sk["out"], non_blocking=True)
                sk["lse_h"].copy_(sk["lse"], non_blocking=True)
            ev_down[i].record(down_s)
        up_s.wait_stream(down_s)
        t1.record(up_s)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1) / n_e2e

    e2e_pass()                                      # warm-up
    e2e_ms = [e2e_pass() for _ in range(2)]
    for sk in sets:                                 # every step's result is the path's result
        st, det = pa.pa_check(plan, sk["ws"], stream)
        if st != 0:
            raise RuntimeError(f"{case.name}: device status {st} ({pa.pa_last_error()})")
    if not torch.equal(sets[0]["out_h"].view(torch.int16), d["out"].cpu().view(torch.int16)):
        raise RuntimeError(f"{case.name}: end-to-end output differs from the device-timed run")
    e2e_step = _max_over_ranks(statistics.mean(e2e_ms), world)

    rec = {"workload": case.name, "desc": synth_desc(cfg), "steps": K, "warmup": args.warmup,
           "ms_per_step": round(ms_max, 5), "kernel_ms": round(run_mean, 5),
           "gpu_launches": launches, "clocks": clk.summary(),
           "kv_bytes_per_step": kv_bytes, "flops_per_step": desc["flops"],
           "items": desc["num_items"], "ctas": desc["num_ctas"], "chunk": desc["chunk"],
           "l2": rotation_note(n_rot, kv_bytes)}
    if flushed_ms is not None:
        rec["flushed"] = {"ms_per_step": round(flushed_ms, 5), "l2": L2_NOTE}
    roof = {"bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": _traffic(case.name),
            "traffic_unit": "bytes per launch (ncu)", "peak_source": peak_kind + " (of measured)"
            if peak_kind.startswith("measured") else peak_kind,
            "kernel": "pa_run attention kernel", "run_ms": round(run_mean, 5),
            "nominal_peak": NOMINAL_PEAK[bound],
            "frac_of_nominal": round(achieved / NOMINAL_PEAK[bound], 4)}
    if kind == "latency":
        # two short sequences: the step is bound by launch latency, so it is
        # reported as a latency; the byte rate is shown for reference only
        rec.update(value=round(ms_max * 1e3, 2), unit="us", higher_is_better=False,
                   e2e={"value": round(e2e_step * 1e3, 2), "unit": "us", "h2d_bytes_per_step": int(h2d),
                        "d2h_bytes_per_step": int(d2h)})
        roof["note"] = "launch-latency bound: the roofline fraction is not meaningful"
    else:
        rec.update(value=round(_job_rate(work, world, ms_max), 2), unit=unit, higher_is_better=True,
                   e2e={"value": round(_job_rate(work, world, e2e_step), 2), "unit": unit,
                        "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                        "mode": "steps back to back: each step's upload and result read overlap "
                                "the neighbouring steps' kernels (two buffer sets, copy streams)",
                        "l2": f"not flushed; steps rotate over {len(caches)} cache "
                              f"cop{'y' if len(caches) == 1 else 'ies'}"})
    rec["roofline"] = roof
    if pool is not None:
        rec["cpu_baseline"] = pool.baseline(case.name, args.cpu_seconds)
    del sets, caches, d, ws, flush
    torch.cuda.empty_cache()
    return rec


def run_cuda(args) -> dict:
    import torch

    rank, world, local = _dist()
    configs = [args.config] if args.config else list(ALL_WORKLOADS)
    cases = {}
    for c in configs:
        case = _workload(c, args.bsz)
        if args.tree_mask:
            from synth.cases import tree_mask
            case.attn_mask = tree_mask(case)
            case.name += " tree-mask"
        if args.fused_merge:
            # another kernel than the two-launch path: its own name keeps the
            # two-launch path's ncu traffic figure off this record
            case.name += " single-launch"
        cases[c] = case
    pool = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pool = CpuPool({c.name: c for c in cases.values()})   # before the first CUDA call
    try:
        torch.cuda.set_device(local)
        dev = torch.device("cuda", local)
        records = {}
        for c in configs:
            records[c] = run_workload(c, cases[c], args, world, local, dev, pool)
    finally:
        if pool is not None:
            pool.close()
    head = records[configs[0]]
    res = {
        "metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": head["higher_is_better"], "scaling": "weak", "vs_baseline": None,
        "dtype": "fp16 (int8 / e4m3 KV dequantised exactly; fp32 accumulate)", "data": "synthetic",
        "config": config_of(configs[0], head, world,
                            {records[c]["workload"]: records[c] for c in configs} if len(configs) > 1 else None),
        "roofline": head["roofline"], "e2e": head["e2e"], "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
    }
    if "cpu_baseline" in head:
        res["cpu_baseline"] = head["cpu_baseline"]
    return res if rank == 0 else None


def config_of(cfg: int, head: dict, world: int, per_workload=None) -> dict:
    """The line's config: the same keys for the CUDA arm and the reference arm."""
    c = {"workload": head["workload"] if head else synth_desc(cfg).split(":")[0],
         "desc": synth_desc(cfg),
         "l2": (head or {}).get("l2", L2_NOTE),
         "parallelism": f"replicas x{world}",
         "algorithmic_unit": "KV bytes of every visible position read once (per token)"
                             if _kind(cfg) != "flops" else
                             "2 (Dqk + Dv) flop per visible (query head, position) pair"}
    if per_workload is not None:
        c["per_workload"] = per_workload
    return c


def run_cache_append(args) -> dict:
    """Times pa_cache_append: the appended tokens of a workload (default the
    append workload's 2.3K tokens x 8 kv heads) quantised into the paged cache.
    Metric: bytes of the bf16 rows read plus cache bytes written, per second."""
    import torch
    import paged_quantized_kv_gqa_gb300 as pa
    from synth.device import to_device
    from synth.cases import new_kv

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    case = _workload(args.config or 3)
    d = to_device(case, dev)
    k, v = new_kv(case)
    kd = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).to(dev)
    vd = None if v is None else torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(dev)
    stride = kd[0].numel()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    plan = pa.pa_plan(pa.problem_of(case), case.seq_lens, case.seq_lens_kv, case.cu_seqlens_q, sms)
    ws = torch.zeros(plan.workspace_size, dtype=torch.uint8, device=dev)
    cargs = pa.make_args(q=d["q"], cache_k=d["cache_k"], cache_v=d["cache_v"],
                         k_scale=d["k_scale"], v_scale=d["v_scale"], block_table=d["block_table"],
                         out=d["out"], lse=d["lse"], seq_lens=d["seq_lens"],
                         seq_lens_kv=d["seq_lens_kv"], cu_seqlens_q=d["cu_seqlens_q"])
    stream = torch.cuda.current_stream(dev)
    pa.pa_plan_upload(plan, ws, stream)
    flush = L2Flush(dev)
    vals = kd.numel() + (0 if vd is None else vd.numel())
    nbytes = vals * 3                      # bf16 read + one stored byte each
    for _ in range(args.warmup):
        flush(1)
        pa.pa_cache_append(plan, cargs, kd, vd, stride, ws, stream)
    st, _ = pa.pa_check(plan, ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {st} ({pa.pa_last_error()})")
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    _barrier(world)
    torch.cuda.synchronize(dev)
    with Clocks(local) as clk:
        for i in range(K):
            flush(i)
            ev[i][0].record(stream)
            pa.pa_cache_append(plan, cargs, kd, vd, stride, ws, stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
    _barrier(world)
    ms = _max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), world)
    work = nbytes / 1e9
    peak, peak_kind = _peaks("hbm")
    # end to end: the new rows up from pinned host memory, the status word back
    kh = kd.cpu().pin_memory()
    vh = None if vd is None else vd.cpu().pin_memory()
    sth = torch.empty(4, dtype=torch.int32).pin_memory()
    e2e_ms = []
    for i in range(max(3, K)):
        flush(i)
        a, b = ev[i % K]
        a.record(stream)
        kd.copy_(kh, non_blocking=True)
        if vd is not None:
            vd.copy_(vh, non_blocking=True)
        pa.pa_cache_append(plan, cargs, kd, vd, stride, ws, stream)
        sth.copy_(ws[:16].view(torch.int32), non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms.append(a.elapsed_time(b))
    e2e = _job_rate(work, world, _max_over_ranks(statistics.mean(e2e_ms), world))
    res = {
        "metric": "KV-cache append (quantise + paged write) GB/s", "value": round(_job_rate(work, world, ms), 2),
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 quotient -> int8 / e4m3 bytes", "data": "synthetic",
        "config": {"workload": case.name + " appended tokens", "tokens": case.total_q,
                   "bytes_per_step": nbytes, "l2": L2_NOTE,
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(work / (ms * 1e-3), 1), "peak": peak,
                     "unit": "GB/s", "frac": round(work / (ms * 1e-3) / peak, 4), "traffic": None,
                     "peak_source": peak_kind, "kernel": "pa_cache_append kernel", "run_ms": round(ms, 5)},
        "e2e": {"value": round(e2e, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(vals * 2), "d2h_bytes_per_step": 16},
        "gpu_launches": K,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import cache_append as ca
        t0 = time.perf_counter()
        sub = synth_subcase(case, max(1, case.bsz // 8))
        sk, sv = new_kv(sub)
        ca.cache_append(sub, sk, sv, sub.cache_k, sub.cache_v if sub.layout != "mla" else None)
        dt = time.perf_counter() - t0
        nb = (sk.size + (0 if sv is None else sv.size)) * 3
        res["cpu_baseline"] = {"value": round(nb / dt / 1e9, 6), "unit": "GB/s", "cores": 1,
                               "kind": "oracle", "sample": f"{sub.total_q} appended tokens "
                               f"({sub.bsz} of {case.bsz} sequences), {dt:.1f} s, numpy"}
    return res if rank == 0 else None


def synth_subcase(case, nseq: int):
    """The first nseq sequences of a workload as a case of its own."""
    import synth
    kw = dict(name=case.name + "-sample", seed=case.seed, seq_lens=case.seq_lens[:nseq],
              seq_lens_kv=case.seq_lens_kv[:nseq], q_heads=case.q_heads, kv_heads=case.kv_heads,
              head_dim_qk=case.head_dim_qk, head_dim_v=case.head_dim_v, kv_dtype=case.kv_dtype,
              scale_kind=case.scale_kind, layout=case.layout, causal=case.causal)
    return synth.make_case(**kw)


def run_reference(args) -> dict:
    """The oracle, as it stands, on the host cores: the reference arm.  Every
    step is a bounded sample of the same workload as the CUDA arm's line."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    cfg = args.config or HEADLINE
    case = _workload(cfg)
    K, W = args.steps, args.warmup
    pool = CpuPool({case.name: case})
    try:
        per = max(2.0, args.cpu_seconds)
        vals = []
        cb = None
        for i in range(W + K):
            cb = pool.baseline(case.name, per)
            if i >= W:
                vals.append(cb["value"])
    finally:
        pool.close()
    v = statistics.mean(vals)
    cb["value"] = round(v, 6)
    unit = cb["unit"]
    return {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": unit,
            "n_gpus": 1, "steps": K, "warmup": W, "higher_is_better": True,
            "ms_per_step": None, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(cfg, {"workload": case.name,
                                                                 "l2": "host CPU run (no GPU L2)"}, 1),
            "cpu_baseline": cb,
            "e2e": {"value": round(v, 6), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=0, choices=[0, 1, 2, 3, 4, 5],
                    help="one workload only (0: all five, decode-2 as the headline)")
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=20.0,
                    help="CPU work (summed over the host cores) of each oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tree-mask", action="store_true",
                    help="speculative verify with a seeded draft-tree mask (decode-family workloads)")
    ap.add_argument("--bsz", type=int, default=0,
                    help="keep only the first BSZ sequences of the workload (same draws): a smaller "
                         "case of the same kernel for profiling captures; not a bench line")
    ap.add_argument("--fused-merge", action="store_true",
                    help="decode-family workloads: merge split rows inside the attention launch "
                         "(opt-in single-launch mode) instead of the separate merge kernel")
    ap.add_argument("--op", default="attention", choices=["attention", "cache-append"],
                    help="attention: the path (default); cache-append: the quantise-and-write "
                         "step before it, on the workload's appended tokens")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if (args.tree_mask or args.bsz or args.fused_merge) and not args.config:
        ap.error("--tree-mask, --bsz and --fused-merge need --config")
    if args.op == "cache-append" and args.impl != "reference":
        res = run_cache_append(args)
    else:
        res = run_reference(args) if args.impl == "reference" else run_cuda(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
