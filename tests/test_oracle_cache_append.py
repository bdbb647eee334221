"""Pins for the oracle of the cache-append step (quantise-and-write of the
appended tokens' K / V), independent of the oracle's own code paths."""
import numpy as np
import pytest
import torch

import synth
from synth.cases import new_kv
from oracle import cache_append as ca
from oracle import attention as oa
from oracle.formats import e4m3_value, int8_value, bf16_to_f64


def test_e4m3_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = np.array([e4m3_value(c) for c in codes], dtype=np.float32)
    assert np.array_equal(ca.e4m3_encode(vals), codes)


def test_e4m3_ties_go_to_even_mantissa_and_saturate():
    # 1.0 = 0x38, 1.125 = 0x39: the midpoint 1.0625 rounds to the even 0x38;
    # 1.1875 (between 0x39 and 0x3A = 1.25) rounds to 0x3A
    assert ca.e4m3_encode(np.float32(1.0625)) == 0x38
    assert ca.e4m3_encode(np.float32(1.1875)) == 0x3A
    # smallest subnormal 2^-9 = 0x01; half of it ties to +0
    assert ca.e4m3_encode(np.float32(2.0 ** -9)) == 0x01
    assert ca.e4m3_encode(np.float32(2.0 ** -10)) == 0x00
    assert ca.e4m3_encode(np.float32(-(2.0 ** -10))) == 0x80   # sign of zero kept
    assert ca.e4m3_encode(np.float32(1000.0)) == 0x7E            # +448
    assert ca.e4m3_encode(np.float32(-1000.0)) == 0xFE           # -448
    assert ca.e4m3_encode(np.float32(464.0)) == 0x7E             # past the top value


def test_e4m3_encode_matches_library_conversion():
    x = (np.random.default_rng(0).standard_normal(50000) * 60).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ca.e4m3_encode(x), ref)


def test_int8_rounds_half_to_even_and_saturates():
    v = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, 127.6, -300.0, 0.49999997],
                 dtype=np.float32)
    got = ca.int8_encode(v).view(np.int8)
    assert got.tolist() == [0, 2, 2, 0, -2, -2, 126, 127, -127, 0]


@pytest.mark.parametrize("kw", [
    dict(kv_dtype="int8", scale_kind="per_kv_head"),
    dict(kv_dtype="int8", scale_kind="per_channel"),
    dict(kv_dtype="fp8_e4m3", scale_kind="per_kv_head"),
])
def test_appended_values_land_in_place_within_half_a_step(kw):
    case = synth.make_case(name="app", seed=5, seq_lens=[70, 3, 0], seq_lens_kv=[100, 0, 9],
                           q_heads=8, kv_heads=2, **kw)
    k, v = new_kv(case)
    ck, cv = ca.cache_append(case, k, v, case.cache_k, case.cache_v)
    table = np.array([(e4m3_value if case.kv_dtype == "fp8_e4m3" else int8_value)(c)
                      for c in range(256)])
    written = np.zeros(ck.shape, bool)
    for b in range(case.bsz):
        lo = int(case.seq_lens_kv[b])
        hi = lo + int(case.seq_lens[b])
        for kvh in range(case.kv_heads):
            # read back through the attention oracle's gather (another code path)
            probe = synth.cases.Case(**{f.name: getattr(case, f.name)
                                        for f in case.__dataclass_fields__.values()})
            probe._cache_k, probe._cache_v = ck, cv
            K, V = oa.gather_raw(probe, b, kvh, hi)
            for which, raw, src in (("k", K, k), ("v", V, v)):
                sc = ca._scales(case, case.k_scale if which == "k" else case.v_scale, kvh, 128)
                x = bf16_to_f64(src[case.cu_seqlens_q[b]:case.cu_seqlens_q[b] + hi - lo, kvh])
                q = x / sc.astype(np.float64)
                back = table[raw[lo:hi]]
                if case.kv_dtype == "int8":
                    inside = np.abs(q) <= 127
                    assert np.all(np.abs(back - q)[inside] <= 0.5 + 1e-6)
                    assert np.all(np.abs(back[~inside]) == 127)
                else:
                    # within half an E4M3 spacing (relative 2^-4) or the subnormal step
                    assert np.all(np.abs(back - q) <= np.maximum(np.abs(q) * 2.0 ** -4, 2.0 ** -10))
    # every byte outside the appended positions is unchanged
    changed_k = ck != case.cache_k
    for b in range(case.bsz):
        for i in range(int(case.seq_lens[b])):
            j = int(case.seq_lens_kv[b]) + i
            changed_k[int(case.block_table[b, j // 64]), :, j % 64, :] = False
    assert not changed_k.any()


def test_mla_rows_are_written_whole():
    case = synth.make_case(name="mla-app", seed=6, seq_lens=[2, 1], seq_lens_kv=[63, 64],
                           q_heads=128, kv_heads=1, head_dim_qk=576, head_dim_v=512,
                           layout="mla", kv_dtype="fp8_e4m3", scale_kind="global")
    k, _ = new_kv(case)
    ck, _ = ca.cache_append(case, k, None, case.cache_k, None)
    s = np.float32(np.asarray(case.k_scale, np.float32).reshape(-1)[0])
    for b in range(case.bsz):
        for i in range(int(case.seq_lens[b])):
            j = int(case.seq_lens_kv[b]) + i
            t = int(case.cu_seqlens_q[b]) + i
            row = ck[int(case.block_table[b, j // 64]), j % 64]
            ref = torch.from_numpy(np.clip(bf16_to_f64(k[t]).astype(np.float32) / s, -448, 448)
                                   ).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(row, ref)
