"""The timeline summaries of paged_quantized_kv_gqa_gb300/trace.py on synthetic
stamps (no GPU): bandwidth over time of the warp-per-item kernel and the
item-boundary periods of the tensor-memory kernel."""
import numpy as np

from paged_quantized_kv_gqa_gb300 import trace


def test_warp_summary_bandwidth_and_finish_times():
    # 2 CTAs x 8 warps, each warp finishes one 8 KB half page every 1 us for 10 us
    tr = np.zeros((2, 10, 16), dtype=np.int64)
    for c in range(2):
        for w in range(8):
            tr[c, :, w] = 1_000_000 + 1000 * np.arange(1, 11)
    text = trace.summarize_warp(tr)
    lines = text.splitlines()
    # 16 warps x 2 half pages per 2 us bin x 8192 bytes / 2 us = 0.13 TB/s
    first_bin = lines[1].split()
    assert first_bin[0] == "0" and abs(float(first_bin[1]) - 0.13) < 0.011
    assert "max 9.0" in lines[-1] and "min 9.0" in lines[-1]


def test_tmem_summary_splits_item_boundaries():
    # one CTA, items of 4 and 4 tiles (128 positions each); P-ready every 1 us
    # inside an item, 3 us for the first tile of the second item
    items = np.zeros((2, 8), dtype=np.int64)
    items[:, 5] = 0
    items[:, 6] = 4 * 128
    ind = np.array([0, 2])
    tr = np.zeros((1, 8, 16), dtype=np.int64)
    t = [0, 1, 2, 3, 6, 7, 8, 9]          # us
    tr[0, :, 4] = 1_000_000 + 1000 * np.array(t)
    tr[0, 3, 10] = tr[0, 4, 4] + 500      # epilogue of item 0 ends 0.5 us after P of tile 4
    text = trace.summarize_tmem(tr, items, ind)
    got = {ln.strip().split(" p10")[0].strip(): ln for ln in text.splitlines()}
    assert "p50 3.00" in got["first tile of an item"]
    assert "p50 1.00" in got["second tile"]
    assert "p50 1.00" in got["tiles inside an item"]
    assert "p50 0.50" in got["item epilogue"]
