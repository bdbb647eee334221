"""Output epilogue of the attention path (oracle side; test infrastructure only).

FastDeploy append_attention_c8_impl.cuh passes shift_bias and smooth_weight
([q_heads * head_dim], activation type) and, for an int8 output, in_scale and
the quant bounds to the step that writes each query row's final output (the
attention kernel for rows with one chunk, the merge for split rows).  The
function that applies them is not on the pages; the reading taken here is the
plainest one their names support:

    v' = (v + shift_bias[h * Dv + d]) * smooth_weight[h * Dv + d]
    bf16 output: bf16_rne(v')
    int8 output: clamp(rint(v' * quant_max_bound * in_scale), quant_min_bound, quant_max_bound)

with v the normalised attention output of query head h, dim d.  The oracle
evaluates v' in float64 from the float64 attention output; the int8 decision
is compared with a tolerance that covers the attention output's own error.
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_to_f64


def apply(out, shift_bits=None, smooth_bits=None):
    """v' for out [T, Hq, Dv] (float64); shift / smooth: bf16 bits [Hq * Dv] or None."""
    T, Hq, Dv = out.shape
    v = np.array(out, dtype=np.float64, copy=True)
    if shift_bits is not None:
        v = v + bf16_to_f64(shift_bits).reshape(Hq, Dv)[None]
    if smooth_bits is not None:
        v = v * bf16_to_f64(smooth_bits).reshape(Hq, Dv)[None]
    return v


def quantize_int8(v, in_scale: float, max_bound: float, min_bound: float) -> np.ndarray:
    """int8 codes of v' (round half to even, clamped to the bounds)."""
    q = np.rint(np.asarray(v, np.float64) * (max_bound * in_scale))
    return np.clip(q, min_bound, max_bound).astype(np.int64)
