"""GPU parity of the decode / speculative-verify path (q_len * G <= 64) against
the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oa
from gpu_helpers import run_case, compare, num_sms
from synth.device import to_device, fill_uniform_i8

pytestmark = pytest.mark.gpu


def test_device_generator_matches_host():
    case = synth.config(2)
    t = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    fill_uniform_i8(t, case.seed, synth.cases.S_K, -127, 127, start=12345)
    host = case.kv_bytes("k", 12345, 1 << 20)
    assert np.array_equal(t.cpu().numpy(), host)


def test_decode_1():
    case = synth.config(1)
    out, lse, plan, _, _ = run_case(case)
    assert plan.describe()["family"] == "decode"
    compare(case, out, lse, label="decode-1")


def test_decode_2_full():
    case = synth.config(2)
    out, lse, plan, _, _ = run_case(case)
    d = plan.describe()
    assert d["chunk"] == 512 and d["max_chunks"] > 1
    compare(case, out, lse, label="decode-2")


def test_spec_verify_4_sampled():
    """Full-size workload 4 in the benchmark's launch configuration; the oracle
    checks a spread of (sequence, kv head) units one by one."""
    case = synth.config(4)
    out, lse, plan, _, _ = run_case(case)
    rng = np.random.default_rng(0)
    bs = sorted(set(rng.choice(case.bsz, 12, replace=False).tolist()) | {0, case.bsz - 1})
    units = [(b, int(rng.integers(case.kv_heads))) for b in bs]
    compare(case, out, lse, units=units, label="spec-verify-4")


EDGE = []
for kv in [0, 1, 62, 63, 64, 65, 127, 128, 129, 511, 512, 513]:
    EDGE.append(dict(seq_lens=[1, 1], seq_lens_kv=[kv, 3], q_heads=8, kv_heads=2, chunk_size=512))
EDGE += [
    dict(seq_lens=[16, 0, 5], seq_lens_kv=[300, 7, 0], q_heads=16, kv_heads=4, chunk_size=128),
    dict(seq_lens=[3, 2], seq_lens_kv=[1000, 1], q_heads=4, kv_heads=4, chunk_size=256),   # G 1
    dict(seq_lens=[8], seq_lens_kv=[700], q_heads=64, kv_heads=8, chunk_size=0),           # G 8, 64 rows
    dict(seq_lens=[4, 4], seq_lens_kv=[90, 200], q_heads=32, kv_heads=4, causal=False, chunk_size=64),
    dict(seq_lens=[1, 1, 1], seq_lens_kv=[40, 2000, 129], q_heads=8, kv_heads=2,
         scale_kind="per_channel", chunk_size=256),
    dict(seq_lens=[2, 3], seq_lens_kv=[333, 64], q_heads=12, kv_heads=4,
         kv_dtype="fp8_e4m3", scale_kind="per_kv_head", chunk_size=128),
    dict(seq_lens=[1, 2], seq_lens_kv=[500, 77], q_heads=8, kv_heads=2, scale_kind="global",
         chunk_size=0),
    dict(seq_lens=[2], seq_lens_kv=[150], q_heads=8, kv_heads=2, chunk_size=0,
         q_stride=(8 + 2 * 2) * 128),                                                       # packed qkv
    dict(seq_lens=[1], seq_lens_kv=[40], q_heads=4, kv_heads=1, chunk_size=0, num_pages=1),  # 1-page pool
    dict(seq_lens=[6] * 3, seq_lens_kv=[2500, 1024, 1023], q_heads=64, kv_heads=8, chunk_size=1024),
]


@pytest.mark.parametrize("kw", EDGE)
def test_decode_edge_cases(kw):
    kw = dict(kw)
    case = synth.make_case(name="edge", seed=7, **kw)
    out, lse, plan, _, _ = run_case(case)
    assert plan.describe()["family"] == "decode"
    compare(case, out, lse, label=str(kw))


@pytest.mark.parametrize("kw", [
    # at most 16 packed rows per tile (warp-per-item kernel), one chunk
    dict(seq_lens=[1, 1], seq_lens_kv=[300, 70], q_heads=8, kv_heads=2, chunk_size=0),
    # 48 packed rows per tile (tensor-memory kernel), one chunk
    dict(seq_lens=[6], seq_lens_kv=[700], q_heads=64, kv_heads=8, chunk_size=0),
])
def test_decode_unaligned_out(kw):
    """The decode family takes an out that is not 16-byte aligned: its kernels
    write whole rows with 16-byte stores only when out allows them."""
    case = synth.make_case(name="unaligned out", seed=11, **kw)
    d = to_device(case)
    flat = torch.zeros(d["out"].numel() + 1, dtype=d["out"].dtype, device=d["out"].device)
    d["out"] = flat[1:].view(d["out"].shape)          # 2 bytes past a 16-byte boundary
    assert d["out"].data_ptr() % 16 != 0
    out, lse, plan, _, _ = run_case(case, d=d)
    assert plan.describe()["family"] == "decode"
    compare(case, out, lse, label="unaligned out " + str(kw))


def test_page_permutation_invariance_bitexact():
    """Same logical cache under two physical page permutations: identical output bits."""
    a = synth.make_case(name="perm", seed=9, seq_lens=[1, 3, 2], seq_lens_kv=[700, 1500, 64],
                        q_heads=16, kv_heads=4, chunk_size=256)
    oa_, la, _, da, _ = run_case(a)
    P = a.num_pages
    perm = np.random.default_rng(3).permutation(P)
    inv = np.argsort(perm)
    b = synth.make_case(name="perm", seed=9, seq_lens=[1, 3, 2], seq_lens_kv=[700, 1500, 64],
                        q_heads=16, kv_heads=4, chunk_size=256)
    b._cache_k = a.cache_k[inv].copy()
    b._cache_v = a.cache_v[inv].copy()
    bt = a.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    b.block_table = bt
    ob, lb, _, _, _ = run_case(b)
    assert np.array_equal(oa_.view(np.uint32), ob.view(np.uint32))
    assert np.array_equal(la.view(np.uint32), lb.view(np.uint32))


def test_repeat_runs_bitexact():
    case = synth.make_case(name="rep", seed=10, seq_lens=[2, 1], seq_lens_kv=[3000, 900],
                           q_heads=32, kv_heads=8, chunk_size=512)
    d = to_device(case)
    o1, l1, _, _, _ = run_case(case, d)
    o2, l2, _, _, _ = run_case(case, d)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_debug_gather_bitexact():
    import paged_quantized_kv_gqa_gb300 as pa
    case = synth.make_case(name="g", seed=12, seq_lens=[2, 1], seq_lens_kv=[200, 70],
                           q_heads=8, kv_heads=2, chunk_size=0)
    d = to_device(case)
    args = pa.make_args(q=d["q"], cache_k=d["cache_k"], cache_v=d["cache_v"],
                        k_scale=d["k_scale"], v_scale=d["v_scale"],
                        block_table=d["block_table"], out=d["out"])
    for b, kvh, pos0, n in [(0, 1, 0, 202), (1, 0, 5, 66), (0, 0, 63, 2)]:
        dk = torch.empty((n, 128), dtype=torch.uint8, device="cuda")
        dv = torch.empty((n, 128), dtype=torch.uint8, device="cuda")
        pa.pa_debug_gather(pa.problem_of(case), args, b, kvh, pos0, n, dk, dv)
        torch.cuda.synchronize()
        K, V = oa.gather_raw(case, b, kvh, pos0 + n)
        assert np.array_equal(dk.cpu().numpy(), K[pos0:])
        assert np.array_equal(dv.cpu().numpy(), V[pos0:])


def test_bad_page_is_reported_not_dereferenced():
    import paged_quantized_kv_gqa_gb300 as pa
    case = synth.make_case(name="bad", seed=13, seq_lens=[1, 1], seq_lens_kv=[100, 100],
                           q_heads=8, kv_heads=2, chunk_size=0)
    d = to_device(case)
    d["block_table"][0, 1] = case.num_pages + 5
    out, lse, plan, _, st = run_case(case, d, check=False)
    assert st == pa.PA_ERR_BAD_PAGE
    # the untouched sequence is still right
    compare(case, out, lse, units=[(1, 0), (1, 1)], label="bad-page neighbour")


def test_bounded_wait_times_out_and_context_survives():
    """A loader that skips its first page load leaves the consumers waiting on a
    barrier nothing completes; the bounded wait must end the kernel with
    PA_ERR_DEVICE_TIMEOUT and leave the context usable."""
    import paged_quantized_kv_gqa_gb300 as pa
    case = synth.make_case(name="to", seed=14, seq_lens=[1], seq_lens_kv=[300], q_heads=8,
                           kv_heads=2, chunk_size=0)
    d = to_device(case)
    pa.pa_debug_set_faults(wait_limit_ns=200_000_000, skip_first_load=True)
    try:
        _, _, _, _, st = run_case(case, d, sms=1, check=False)
    finally:
        pa.pa_debug_set_faults(0, False)
    assert st == pa.PA_ERR_DEVICE_TIMEOUT
    out, lse, _, _, st2 = run_case(case, d)
    assert st2 == 0
    compare(case, out, lse, label="after timeout")
