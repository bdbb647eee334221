"""Plain fp64 CPU oracle for paged, quantised-KV attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes anything under ``oracle/``; only ``tests/``, ``__graft_entry__.smoke``
and the CPU-baseline leg of ``bench.py`` do.  The oracle shares no code, table
or constant with the CUDA path: it decodes the cache formats, gathers through
the block table and evaluates the masked softmax directly, in float64, from the
definition of the operation on the source pages (FastDeploy
append_attention_c8_impl.cuh, multi_query_append_attention_c8_kernel and its
warp1_4 decode variant; FlashInfer persistent.cuh, the state merge; XQA
mla_sm120.cu, kernel_mha and mergePartialOutputs).

Modules:
  formats   - int8 and OCP FP8 E4M3 decoding, bf16 bit decoding
  attention - exact attention per (sequence, kv head); per-chunk partial states
              and their log-sum-exp merge
  planner   - an independent implementation of the work-item planner spec, used
              to check the production planner bit for bit

Parity status: every function here is pinned by tests in tests/test_oracle.py
(closed forms, invariants, brute force and library special cases).
"""
from . import formats, attention, planner  # noqa: F401
