"""Places a synthetic Case in device memory (torch tensors).

Uniform int8 caches are generated directly on the device by
``synth/libpa_synth.so`` (the same counter formulas as synth.rng, so every
byte equals the host draw); everything else is copied from the host arrays.
Holds no attention arithmetic.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpa_synth.so")
_lib = None


def _synth_lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB):
            raise ImportError(f"{_LIB} missing: build it with __graft_entry__.build()")
        _lib = ctypes.CDLL(_LIB)
        _lib.synth_fill_uniform_i8.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                               ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int32,
                                               ctypes.c_int32, ctypes.c_void_p]
        _lib.synth_fill_uniform_i8.restype = ctypes.c_int
    return _lib


def fill_uniform_i8(t: torch.Tensor, seed: int, stream_id: int, lo: int, hi: int, start: int = 0):
    """Fill a uint8 CUDA tensor with the host generator's uniform int8 draws."""
    assert t.is_cuda and t.dtype == torch.uint8 and t.is_contiguous()
    s = torch.cuda.current_stream(t.device).cuda_stream
    rc = _synth_lib().synth_fill_uniform_i8(t.data_ptr(), start, t.numel(), seed, stream_id, lo, hi, s)
    if rc != 0:
        raise RuntimeError(f"synth_fill_uniform_i8 failed ({rc})")


def to_device(case, device="cuda", generate_on_device=True) -> dict:
    """Return torch tensors for every input of the case plus zeroed out / lse."""
    from .cases import S_K, S_V, INT8, MLA
    dev = torch.device(device)
    T = case.total_q
    d = {}
    d["q"] = torch.from_numpy(case.q_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    if case.kv_dtype == INT8 and generate_on_device and case._cache_k is None:
        lo, hi = case.int8_range
        k = torch.empty(case.k_shape, dtype=torch.uint8, device=dev)
        fill_uniform_i8(k, case.seed, S_K, lo, hi)
        if case.layout == MLA:
            v = k
        else:
            v = torch.empty(case.v_shape, dtype=torch.uint8, device=dev)
            fill_uniform_i8(v, case.seed, S_V, lo, hi)
    else:
        k = torch.from_numpy(np.ascontiguousarray(case.cache_k)).to(dev)
        v = k if case.layout == MLA else torch.from_numpy(np.ascontiguousarray(case.cache_v)).to(dev)
    d["cache_k"], d["cache_v"] = k, v
    if case.scale_kind == "global":
        d["k_scale"] = torch.from_numpy(np.asarray(case.k_scale, np.float32)).to(dev)
        d["v_scale"] = torch.from_numpy(np.asarray(case.v_scale, np.float32)).to(dev)
    else:
        d["k_scale"] = torch.from_numpy(case.k_scale.view(np.int16)).view(torch.bfloat16).to(dev)
        d["v_scale"] = torch.from_numpy(case.v_scale.view(np.int16)).view(torch.bfloat16).to(dev)
    d["block_table"] = torch.from_numpy(case.block_table).to(dev)
    d["seq_lens"] = torch.from_numpy(case.seq_lens).to(dev)
    d["seq_lens_kv"] = torch.from_numpy(case.seq_lens_kv).to(dev)
    d["cu_seqlens_q"] = torch.from_numpy(case.cu_seqlens_q).to(dev)
    d["out"] = torch.zeros((T, case.q_heads, case.head_dim_v), dtype=torch.bfloat16, device=dev)
    d["lse"] = torch.zeros((T, case.q_heads), dtype=torch.float32, device=dev)
    if getattr(case, "attn_mask", None) is not None:
        d["attn_mask"] = torch.from_numpy(np.ascontiguousarray(case.attn_mask, np.uint8)).to(dev)
    return d
