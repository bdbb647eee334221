"""Paged, quantised-KV GQA / MLA attention on GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/pa.h`` (``libpa_gb300.so``,
built in-tree by ``paged_quantized_kv_gqa_gb300.build``).  The functions keep
the C names: pa_plan, pa_plan_upload, pa_run, pa_merge, pa_check,
pa_debug_gather, pa_debug_set_faults.  They only marshal arguments; every step
of the attention runs in the library's CUDA kernels.  There is no fallback:
importing this package fails if the library has not been built.

Device buffers may be given as torch tensors (their data_ptr is used) or as
raw integer addresses; streams as torch.cuda.Stream, raw integers or None (the
current torch stream when torch has CUDA, else the legacy default stream).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# PA_GB300_TRACE=1 selects the library built with the pipeline trace (the
# trace module sets it); PA_GB300_DEBUG=1 the debug library (work-item bounds
# checks, poisoned shared and tensor memory); the default library has neither
LIB_PATH = os.path.join(_HERE, "libpa_gb300_trace.so" if os.environ.get("PA_GB300_TRACE") == "1"
                        else "libpa_gb300_debug.so" if os.environ.get("PA_GB300_DEBUG") == "1"
                        else "libpa_gb300.so")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA = 0, 1, 2, 3
PA_ERR_DEVICE_TIMEOUT, PA_ERR_BAD_PAGE, PA_ERR_BAD_ITEM = 4, 5, 6
KV_DTYPES = {"int8": 0, "fp8_e4m3": 1}
SCALE_KINDS = {"per_kv_head": 0, "per_channel": 1, "global": 2}
LAYOUTS = {"gqa": 0, "mla": 1}
FAMILIES = {0: "decode", 1: "append", 2: "mla"}


class PaProblem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "bsz", "q_heads", "kv_heads", "head_dim_qk", "head_dim_v", "block_size",
        "max_blocks_per_seq", "num_pages", "kv_dtype", "scale_kind", "layout", "causal",
        "chunk_size")] + [("sm_scale", ctypes.c_float), ("q_stride", ctypes.c_int64)]


class PaArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "q", "cache_k", "cache_v", "k_scale", "v_scale", "block_table", "seq_lens",
        "seq_lens_kv", "cu_seqlens_q", "out", "lse", "attn_mask", "shift_bias",
        "smooth_weight")] + [("out_int8", ctypes.c_int32), ("in_scale", ctypes.c_float),
                             ("quant_max_bound", ctypes.c_float),
                             ("quant_min_bound", ctypes.c_float)]


class PaPlanDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "family", "chunk_size", "tokens_per_tile", "num_items", "num_ctas", "total_q",
        "max_chunks", "n_merge")] + [
        ("items", ctypes.POINTER(ctypes.c_int32)),
        ("work_indptr", ctypes.POINTER(ctypes.c_int32)),
        ("nch_token", ctypes.POINTER(ctypes.c_int32)),
        ("merge_tokens", ctypes.POINTER(ctypes.c_int32)),
        ("workspace_bytes", ctypes.c_size_t),
        ("kv_bytes", ctypes.c_int64),
        ("flops", ctypes.c_double),
        ("fused_merge", ctypes.c_int32),
        ("plan_bytes", ctypes.c_size_t)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    P32 = ctypes.POINTER(ctypes.c_int32)
    sig = {
        "pa_plan": ([ctypes.POINTER(PaProblem), P32, P32, P32, i32, ctypes.POINTER(vp)], i32),
        "pa_plan_describe": ([vp, ctypes.POINTER(PaPlanDesc)], i32),
        "pa_workspace_size": ([vp], ctypes.c_size_t),
        "pa_plan_upload": ([vp, vp, vp], i32),
        "pa_run": ([vp, ctypes.POINTER(PaArgs), vp, vp], i32),
        "pa_merge": ([vp, ctypes.POINTER(PaArgs), vp, vp], i32),
        "pa_check": ([vp, vp, vp, P32], i32),
        "pa_plan_destroy": ([vp], None),
        "pa_last_error": ([], ctypes.c_char_p),
        "pa_debug_gather": ([ctypes.POINTER(PaProblem), ctypes.POINTER(PaArgs), i32, i32, i32,
                             i32, vp, vp, vp], i32),
        "pa_debug_set_faults": ([i64, i32], i32),
        "pa_run_static": ([vp, ctypes.POINTER(PaArgs), vp, i32], i32),
        "pa_debug_set_trace": ([vp, i32, i32], i32),
        "pa_set_fused_merge": ([i32], i32),
        "pa_cache_append": ([vp, ctypes.POINTER(PaArgs), vp, vp, i64, vp, vp], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


lib = _load()


class PaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"pa status {status}: {msg}")
        self.status = status


def _check(status: int):
    if status != PA_OK:
        raise PaError(status, lib.pa_last_error().decode(errors="replace"))


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> Optional[int]:
    if s is None:
        try:
            import torch
            if torch.cuda.is_available():
                return int(torch.cuda.current_stream().cuda_stream)
        except Exception:  # pragma: no cover - torch without CUDA
            pass
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def make_problem(*, bsz, q_heads, kv_heads, head_dim_qk, head_dim_v, block_size,
                 max_blocks_per_seq, num_pages, kv_dtype, scale_kind, layout, causal,
                 chunk_size, sm_scale, q_stride) -> PaProblem:
    p = PaProblem()
    p.bsz, p.q_heads, p.kv_heads = bsz, q_heads, kv_heads
    p.head_dim_qk, p.head_dim_v, p.block_size = head_dim_qk, head_dim_v, block_size
    p.max_blocks_per_seq, p.num_pages = max_blocks_per_seq, num_pages
    p.kv_dtype = KV_DTYPES[kv_dtype] if isinstance(kv_dtype, str) else kv_dtype
    p.scale_kind = SCALE_KINDS[scale_kind] if isinstance(scale_kind, str) else scale_kind
    p.layout = LAYOUTS[layout] if isinstance(layout, str) else layout
    p.causal = int(bool(causal))
    p.chunk_size = chunk_size
    p.sm_scale = sm_scale
    p.q_stride = q_stride
    return p


def problem_of(case) -> PaProblem:
    """PaProblem from any object carrying the problem fields (e.g. synth.Case)."""
    return make_problem(bsz=case.bsz, q_heads=case.q_heads, kv_heads=case.kv_heads,
                        head_dim_qk=case.head_dim_qk, head_dim_v=case.head_dim_v,
                        block_size=case.block_size, max_blocks_per_seq=case.max_blocks_per_seq,
                        num_pages=case.num_pages, kv_dtype=case.kv_dtype,
                        scale_kind=case.scale_kind, layout=case.layout, causal=case.causal,
                        chunk_size=case.chunk_size, sm_scale=case.sm_scale,
                        q_stride=case.q_stride)


class Plan:
    """Owns a pa_plan_t handle."""

    def __init__(self, handle: int, problem: PaProblem):
        self.handle = handle
        self.problem = problem

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h:
            lib.pa_plan_destroy(h)

    def describe(self) -> dict:
        d = PaPlanDesc()
        _check(lib.pa_plan_describe(self.handle, ctypes.byref(d)))
        arr = lambda p, n: np.ctypeslib.as_array(p, shape=(n,)).copy() if n else np.zeros(0, np.int32)
        return dict(family=FAMILIES[d.family], chunk=d.chunk_size,
                    tokens_per_tile=d.tokens_per_tile, num_items=d.num_items,
                    num_ctas=d.num_ctas, total_q=d.total_q, max_chunks=d.max_chunks,
                    items=arr(d.items, d.num_items * 8).reshape(-1, 8),
                    work_indptr=arr(d.work_indptr, d.num_ctas + 1),
                    nch_token=arr(d.nch_token, d.total_q),
                    merge_tokens=arr(d.merge_tokens, d.n_merge),
                    workspace_bytes=int(d.workspace_bytes), kv_bytes=int(d.kv_bytes),
                    flops=float(d.flops), fused_merge=bool(d.fused_merge),
                    plan_bytes=int(d.plan_bytes))

    @property
    def workspace_size(self) -> int:
        return int(lib.pa_workspace_size(self.handle))


def pa_plan(problem: PaProblem, seq_lens, seq_lens_kv, cu_seqlens_q, num_sms: int) -> Plan:
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    sk = np.ascontiguousarray(seq_lens_kv, dtype=np.int32)
    cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    P32 = ctypes.POINTER(ctypes.c_int32)
    h = ctypes.c_void_p()
    _check(lib.pa_plan(ctypes.byref(problem), sl.ctypes.data_as(P32), sk.ctypes.data_as(P32),
                       cu.ctypes.data_as(P32), int(num_sms), ctypes.byref(h)))
    return Plan(h.value, problem)


def make_args(*, q, cache_k, cache_v, k_scale, v_scale, block_table, out, lse=None,
              seq_lens=None, seq_lens_kv=None, cu_seqlens_q=None, attn_mask=None,
              shift_bias=None, smooth_weight=None, out_int8=False, in_scale=1.0,
              quant_max_bound=127.0, quant_min_bound=-127.0) -> PaArgs:
    a = PaArgs()
    a.q, a.cache_k, a.cache_v = _ptr(q), _ptr(cache_k), _ptr(cache_v)
    a.k_scale, a.v_scale, a.block_table = _ptr(k_scale), _ptr(v_scale), _ptr(block_table)
    a.seq_lens, a.seq_lens_kv, a.cu_seqlens_q = _ptr(seq_lens), _ptr(seq_lens_kv), _ptr(cu_seqlens_q)
    a.out, a.lse = _ptr(out), _ptr(lse)
    a.attn_mask = _ptr(attn_mask)
    a.shift_bias, a.smooth_weight = _ptr(shift_bias), _ptr(smooth_weight)
    a.out_int8 = 1 if out_int8 else 0
    a.in_scale, a.quant_max_bound, a.quant_min_bound = in_scale, quant_max_bound, quant_min_bound
    return a


def pa_plan_upload(plan: Plan, workspace, stream=None):
    _check(lib.pa_plan_upload(plan.handle, _ptr(workspace), _stream(stream)))


def pa_run(plan: Plan, args: PaArgs, workspace, stream=None):
    _check(lib.pa_run(plan.handle, ctypes.byref(args), _ptr(workspace), _stream(stream)))


def pa_merge(plan: Plan, args: PaArgs, workspace, stream=None):
    _check(lib.pa_merge(plan.handle, ctypes.byref(args), _ptr(workspace), _stream(stream)))


def pa_check(plan: Optional[Plan], workspace, stream=None):
    """Synchronises the stream; returns (status, detail) of the workspace status word."""
    detail = ctypes.c_int32(0)
    st = lib.pa_check(plan.handle if plan else None, _ptr(workspace), _stream(stream),
                      ctypes.byref(detail))
    return int(st), int(detail.value)


def pa_debug_gather(problem: PaProblem, args: PaArgs, b: int, kv_head: int, pos0: int, n: int,
                    dst_k, dst_v, stream=None):
    _check(lib.pa_debug_gather(ctypes.byref(problem), ctypes.byref(args), b, kv_head, pos0, n,
                               _ptr(dst_k), _ptr(dst_v), _stream(stream)))


def pa_debug_set_faults(wait_limit_ns: int = 0, skip_first_load: bool = False):
    _check(lib.pa_debug_set_faults(int(wait_limit_ns), int(bool(skip_first_load))))


def pa_run_static(plan: Plan, args: PaArgs, stream=None, check: bool = False):
    """Upload, run and merge with the library's built-in 32 MiB device workspace
    (for callers that cannot allocate device memory; see include/pa.h).
    check=True synchronises the stream and raises on a device-side error."""
    _check(lib.pa_run_static(plan.handle, ctypes.byref(args), _stream(stream), int(bool(check))))


def pa_cache_append(plan: Plan, args: PaArgs, k_new, v_new, kv_stride: int, workspace,
                    stream=None):
    """Quantise the appended tokens' K / V rows (bf16, token stride kv_stride
    elements) into the paged cache of args (see include/pa.h)."""
    _check(lib.pa_cache_append(plan.handle, ctypes.byref(args), _ptr(k_new), _ptr(v_new),
                               int(kv_stride), _ptr(workspace), _stream(stream)))


def pa_debug_set_trace(buf=None, ctas: int = 0, tiles_per_cta: int = 0):
    """Enable (device uint64 buffer of ctas * tiles_per_cta * 16) or disable (None)
    the kernels' %globaltimer pipeline trace (traced library only: see
    PA_GB300_TRACE; the default library raises PA_ERR_UNSUPPORTED)."""
    _check(lib.pa_debug_set_trace(_ptr(buf), int(ctas), int(tiles_per_cta)))


def pa_set_fused_merge(on: bool):
    """Decode-family plans built afterwards merge split rows inside pa_run (True)
    or leave them to pa_merge's separate kernel (False, the default)."""
    _check(lib.pa_set_fused_merge(1 if on else 0))


def pa_last_error() -> str:
    return lib.pa_last_error().decode(errors="replace")
