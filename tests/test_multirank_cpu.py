"""Multi-rank host logic on CPU (gloo, world size 2).

The path shards by sequence with no exchange, so the benchmark runs one
independent replica per GPU and only needs max-over-ranks timing; a
context-parallel split of one long sequence would add one exchange (gather the
(o, m, d) partial states of each rank's KV range, then merge).  Both are
exercised here among CPU processes, never across GPUs.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import synth
        from oracle import attention as oa

        # (1) replicas: the job is charged the slowest rank's time
        ms = [1.5, 2.5][rank]
        ms_max = bench._max_over_ranks(ms, world, device="cpu")
        rate = bench._job_rate(10.0, world, ms_max)

        # (2) context parallel: each rank owns half of the KV positions of one
        # sequence, computes its partial state, the states are all-gathered
        case = synth.make_case(name="cp", seed=31, seq_lens=[3], seq_lens_kv=[500],
                               q_heads=8, kv_heads=2)
        kvtot = int(case.seq_lens_kv[0] + case.seq_lens[0])
        half = (kvtot // 2) // case.block_size * case.block_size
        bounds = [(0, half), (half, kvtot)][rank]
        outs = []
        for kvh in range(case.kv_heads):
            M, Dn, O = oa.unit_partials(case, 0, kvh, [bounds])
            parts = [torch.from_numpy(np.ascontiguousarray(a)) for a in (M, Dn, O)]
            gathered = []
            for t in parts:
                buf = [torch.empty_like(t) for _ in range(world)]
                dist.all_gather(buf, t)
                gathered.append(torch.cat(buf, dim=0).numpy())
            out, lse = oa.merge_states(*gathered)
            ref_o, ref_l = oa.unit_attention(case, 0, kvh)
            outs.append((float(np.abs(out - ref_o).max()), float(np.abs(lse - ref_l).max())))
        q.put((rank, ms_max, rate, outs))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_replicas_and_partial_exchange():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, rate, outs in res:
        assert ms_max == 2.5                       # max over ranks, seen by every rank
        assert rate == pytest.approx(10.0 * 2 / 2.5e-3)
        for err_o, err_l in outs:
            assert err_o < 1e-12 and err_l < 1e-12  # exchange + merge == unsplit
