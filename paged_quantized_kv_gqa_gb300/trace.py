"""Pipeline timeline of one pa_run on a synthetic workload (diagnostics).

    python -m paged_quantized_kv_gqa_gb300.trace --config 2
    python -m paged_quantized_kv_gqa_gb300.trace --config 4

Builds (if needed) and loads the traced library (libpa_gb300_trace.so: the
kernels compiled with PA_TRACE), runs the workload's attention kernel a few
times, then once with the %globaltimer trace of pa_debug_set_trace enabled,
and prints a summary:

  * decode tiles of at most 16 packed rows (warp-per-item kernel): the KV bytes
    the kernel consumed per 2 us of the launch (a bandwidth-over-time profile)
    and when the warps finished;
  * the tensor-memory decode kernel: the time between consecutive P-ready
    events of a CTA, split into the first and second tile of an item and the
    tiles inside an item, and the item epilogue's duration.

The traced launch is slower than a plain one (its stamps are global stores);
compare the shape, not the absolute time.  Needs a GPU and the built library.
"""
import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _tiles(items, ind, c, tile):
    return int(sum((items[it, 6] - items[it, 5] + tile - 1) // tile for it in range(ind[c], ind[c + 1])))


def _pct(v):
    v = np.asarray(v, dtype=np.float64) / 1e3
    return "p10 %.2f  p50 %.2f  p90 %.2f  mean %.2f us" % (*np.percentile(v, [10, 50, 90]), v.mean())


def summarize_warp(tr, bytes_per_stage=8192, warps=8, bin_us=2.0):
    """Bandwidth over time of the warp-per-item kernel (events 0..warps-1 =
    a warp finished a half page)."""
    done = tr[:, :, :warps].reshape(-1)
    t0 = done[done > 0].min()
    done = (done[done > 0] - t0) / 1e3
    edges = np.arange(0.0, done.max() + bin_us, bin_us)
    hist, _ = np.histogram(done, edges)
    lines = ["  t (us)   TB/s"]
    for e, n in zip(edges, hist):
        rate = n * bytes_per_stage / (bin_us * 1e-6) / 1e12
        lines.append("  %6.0f  %5.2f  %s" % (e, rate, "#" * int(rate * 8)))
    ends = []
    for c in range(tr.shape[0]):
        for w in range(warps):
            d = tr[c, :, w]
            d = d[d > 0]
            if len(d):
                ends.append((d.max() - t0) / 1e3)
    e = np.array(ends)
    lines.append("  warps finished: min %.1f  p10 %.1f  p50 %.1f  p90 %.1f  max %.1f us"
                 % (e.min(), *np.percentile(e, [10, 50, 90]), e.max()))
    return "\n".join(lines)


def summarize_tmem(tr, items, ind, tile=128):
    """P-ready periods (event 4) at item boundaries and inside items, and the
    item epilogue (event 10 of the last tile minus event 4 of the next)."""
    first, second, inside, epi = [], [], [], []
    for c in range(tr.shape[0]):
        n, last = 0, []
        for it in range(ind[c], ind[c + 1]):
            n += (items[it, 6] - items[it, 5] + tile - 1) // tile
            last.append(n - 1)
        n = min(n, tr.shape[1])
        ends = set(last)
        p4 = tr[c, :n, 4]
        for g in range(1, n):
            if p4[g] <= 0 or p4[g - 1] <= 0:
                continue
            d = p4[g] - p4[g - 1]
            (first if g - 1 in ends else second if g - 2 in ends else inside).append(d)
        for gl in last[:-1]:
            if gl + 1 < n and tr[c, gl, 10] > 0 and tr[c, gl + 1, 4] > 0:
                epi.append(tr[c, gl, 10] - tr[c, gl + 1, 4])
    out = []
    for name, v in (("first tile of an item", first), ("second tile", second),
                    ("tiles inside an item", inside), ("item epilogue", epi)):
        if v:
            out.append("  %-22s %s  (n=%d)" % (name, _pct(v), len(v)))
    return "\n".join(out)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--config", type=int, default=2, choices=[2, 4])
    ap.add_argument("--bsz", type=int, default=0, help="keep only the first BSZ sequences")
    ap.add_argument("--save", default="", help="also write the raw stamps to this .npz file")
    args = ap.parse_args()

    if os.environ.get("PA_GB300_TRACE") != "1":
        # the package loads its library on import: build the traced one and
        # start again with it selected
        import importlib.util
        spec = importlib.util.spec_from_file_location(
            "pa_build", os.path.join(ROOT, "paged_quantized_kv_gqa_gb300", "build.py"))
        bmod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(bmod)
        bmod.build(trace=True)
        os.environ["PA_GB300_TRACE"] = "1"
        os.execv(sys.executable, [sys.executable, "-m", "paged_quantized_kv_gqa_gb300.trace", *sys.argv[1:]])

    import torch
    import synth
    import paged_quantized_kv_gqa_gb300 as pa
    from synth.device import to_device

    case = synth.config(args.config, args.bsz)
    dev = torch.device("cuda", 0)
    d = to_device(case, dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    plan = pa.pa_plan(pa.problem_of(case), case.seq_lens, case.seq_lens_kv, case.cu_seqlens_q, sms)
    desc = plan.describe()
    ws = torch.zeros(plan.workspace_size, dtype=torch.uint8, device=dev)
    cargs = pa.make_args(q=d["q"], cache_k=d["cache_k"], cache_v=d["cache_v"], k_scale=d["k_scale"],
                         v_scale=d["v_scale"], block_table=d["block_table"], out=d["out"], lse=d["lse"],
                         attn_mask=d.get("attn_mask"))
    pa.pa_plan_upload(plan, ws)
    warp_kernel = int(np.max(case.seq_lens)) * case.group <= 16 and not desc["fused_merge"]
    tile = 32 if warp_kernel else 128           # half pages / 128-position tiles
    # L2 is emptied before each launch: a 512 MiB write, then a 256 MiB read
    # that writes the dirty lines back before the launch starts
    wbuf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    rbuf = torch.ones(32 << 20, dtype=torch.int64, device=dev)
    sink = torch.empty(1, dtype=torch.int64, device=dev)

    def flush(v):
        wbuf.fill_(v)
        sink.copy_(rbuf.sum().view(1))

    for i in range(3):
        flush(i)
        pa.pa_run(plan, cargs, ws)
    items = np.array(desc["items"]).reshape(-1, 8)
    ind = np.array(desc["work_indptr"])
    ctas = desc["num_ctas"]
    tiles = max(_tiles(items, ind, c, tile) for c in range(ctas))
    buf = torch.zeros(ctas * tiles * 16, dtype=torch.int64, device=dev)
    pa.pa_debug_set_trace(buf, ctas, tiles)
    flush(7)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    pa.pa_run(plan, cargs, ws)
    e1.record()
    torch.cuda.synchronize()
    pa.pa_debug_set_trace(None, 0, 0)
    st, _ = pa.pa_check(plan, ws)
    if st != 0:
        raise SystemExit(f"device status {st}: {pa.pa_last_error()}")
    tr = buf.cpu().numpy().reshape(ctas, tiles, 16).astype(np.int64)
    print(f"{case.name}: traced launch {e0.elapsed_time(e1) * 1e3:.1f} us, {ctas} CTAs, "
          f"{'warp-per-item' if warp_kernel else 'tensor-memory'} decode kernel")
    print(summarize_warp(tr) if warp_kernel else summarize_tmem(tr, items, ind))
    if args.save:
        np.savez_compressed(args.save, trace=tr, items=items, indptr=ind)


if __name__ == "__main__":
    main()
