"""Cases for the debug library (kernels compiled with PA_DEBUG: work-item
bounds checks, shared and tensor memory filled with NaN bytes before first
use).  Run as a script in a process with PA_GB300_DEBUG=1, which makes the
binding load libpa_gb300_debug.so; tests/test_gpu_debug_build.py does that.

1. Small cases of every kernel family (warp-per-item decode, tensor-memory
   decode at 32 and 48 rows, per-channel scales, fp8, a draft-tree mask,
   append, MLA with fixed chunks and with page shares) against the fp64
   oracle: a kernel that read shared or tensor memory it never wrote would
   carry the poison into its output as NaN.
2. One plan whose first item of a sequence with 2 of the plan's 3 chunks gets
   chunk index 2 (its own chunk count), written into the uploaded workspace:
   the item check reports PA_ERR_BAD_ITEM with that item's index, and a clean
   run afterwards reports PA_OK.  Even unchecked, that item would only write
   the token's unused third partial slot, inside the workspace.

Exits non-zero on the first failure."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402
from synth.cases import tree_mask  # noqa: E402
from synth.device import to_device  # noqa: E402
import paged_quantized_kv_gqa_gb300 as pa  # noqa: E402
from gpu_helpers import run_case, compare, num_sms  # noqa: E402

MLA = dict(q_heads=128, kv_heads=1, head_dim_qk=576, head_dim_v=512, layout="mla",
           scale_kind="global", sm_scale=1.0 / np.sqrt(192.0), kv_dtype="fp8_e4m3")

CASES = [
    ("decode warp-per-item, split", "decode",
     dict(seq_lens=[1, 1], seq_lens_kv=[1500, 3], q_heads=8, kv_heads=2, chunk_size=512)),
    ("decode 48 rows, split", "decode",
     dict(seq_lens=[6, 6], seq_lens_kv=[1500, 300], q_heads=64, kv_heads=8, chunk_size=512)),
    ("decode 32 rows, per-channel", "decode",
     dict(seq_lens=[4], seq_lens_kv=[900], q_heads=64, kv_heads=8, scale_kind="per_channel",
          chunk_size=0)),
    ("decode fp8, split", "decode",
     dict(seq_lens=[8, 5, 1], seq_lens_kv=[200, 7, 63], q_heads=32, kv_heads=4, chunk_size=64,
          kv_dtype="fp8_e4m3")),
    ("append", "append",
     dict(seq_lens=[150, 70], seq_lens_kv=[400, 33], q_heads=32, kv_heads=8, kv_dtype="fp8_e4m3")),
    ("mla, split", "mla", dict(MLA, seq_lens=[2, 1, 2], seq_lens_kv=[700, 1000, 129], chunk_size=256)),
    ("mla, page shares", "mla", dict(MLA, seq_lens=[1, 2], seq_lens_kv=[3000, 2500], chunk_size=-1)),
]


def parity():
    for i, (label, family, kw) in enumerate(CASES):
        case = synth.make_case(name="debug " + label, seed=40 + i, **kw)
        out, lse, plan, _, _ = run_case(case)
        assert plan.describe()["family"] == family, (label, plan.describe()["family"])
        compare(case, out, lse, label=label)
    case = synth.make_case(name="debug tree", seed=50, seq_lens=[6, 6, 3], seq_lens_kv=[500, 64, 1000],
                           q_heads=64, kv_heads=8, chunk_size=128)
    case.attn_mask = tree_mask(case)
    out, lse, _, _, _ = run_case(case)
    compare(case, out, lse, label="decode tree mask")


def bad_item():
    case = synth.make_case(name="debug bad item", seed=51, seq_lens=[1, 1], seq_lens_kv=[1500, 700],
                           q_heads=8, kv_heads=2, chunk_size=512)
    d = to_device(case)
    plan = pa.pa_plan(pa.problem_of(case), case.seq_lens, case.seq_lens_kv, case.cu_seqlens_q, num_sms())
    desc = plan.describe()
    items = desc["items"]
    nchs = items[:, 7] >> 16
    assert desc["max_chunks"] == 3
    k = int(np.nonzero(nchs == 2)[0][0])
    ws = torch.zeros(max(plan.workspace_size, 256), dtype=torch.uint8, device="cuda")
    args = pa.make_args(q=d["q"], cache_k=d["cache_k"], cache_v=d["cache_v"], k_scale=d["k_scale"],
                        v_scale=d["v_scale"], block_table=d["block_table"], out=d["out"], lse=d["lse"],
                        seq_lens=d["seq_lens"], seq_lens_kv=d["seq_lens_kv"],
                        cu_seqlens_q=d["cu_seqlens_q"])
    pa.pa_plan_upload(plan, ws)
    torch.cuda.synchronize()
    good = ws.cpu().numpy().view(np.int32).copy()
    # the item's record in the uploaded plan (the items are stored in order)
    win = np.lib.stride_tricks.sliding_window_view(good, 8)
    pos = np.nonzero((win == items[k]).all(axis=1))[0]
    assert len(pos) >= 1, "item record not found in the workspace"
    nch = int(items[k, 7]) >> 16
    bad = good.copy()
    bad[pos[0] + 7] = nch | (nch << 16)
    ws.copy_(torch.from_numpy(bad.view(np.uint8)).to(ws.device))
    torch.cuda.synchronize()
    pa.pa_run(plan, args, ws)
    st, det = pa.pa_check(plan, ws)
    assert st == pa.PA_ERR_BAD_ITEM and det == k, (st, det, k)
    ws.copy_(torch.from_numpy(good.view(np.uint8)).to(ws.device))
    torch.cuda.synchronize()
    pa.pa_run(plan, args, ws)
    pa.pa_merge(plan, args, ws)
    st, det = pa.pa_check(plan, ws)
    assert st == pa.PA_OK, (st, det)
    compare(case, d["out"].float().cpu().numpy(), d["lse"].cpu().numpy(), label="after the bad item")


if __name__ == "__main__":
    print("library", os.path.basename(pa.LIB_PATH))
    assert os.path.basename(pa.LIB_PATH) == "libpa_gb300_debug.so", pa.LIB_PATH
    parity()
    bad_item()
    print("debug library: all cases passed")
