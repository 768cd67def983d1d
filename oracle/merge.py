"""Split-result merge definition -- TEST INFRASTRUCTURE ONLY.

When the tokens of one row are partitioned into chunks, each chunk s yields a
normalised partial output o_s and its log-sum-exp lse_s.  The exact result of
the whole row is

    M   = max_s lse_s
    w_s = exp(lse_s - M)
    out = sum_s w_s * o_s / sum_s w_s,     lse = M + ln(sum_s w_s)

(the pages only name "partial" kernels -- 1Cat-vLLM PR #647, Fix -- and leave
the merge unstated; this is the standard log-sum-exp identity for softmax).
A chunk with no visible token has lse = -inf and weight 0; if every chunk is
empty the row is out = 0, lse = -inf.
"""
from __future__ import annotations

import numpy as np


def lse_merge(o_parts, lse_parts):
    o = np.asarray(o_parts, dtype=np.float64)
    lse = np.asarray(lse_parts, dtype=np.float64)
    M = np.max(lse, axis=0)
    empty = ~np.isfinite(M)
    Ms = np.where(empty, 0.0, M)
    w = np.exp(lse - Ms)
    den = np.sum(w, axis=0)
    num = np.sum(w[..., None] * o, axis=0) if o.ndim == lse.ndim + 1 else np.sum(w * o, axis=0)
    with np.errstate(invalid="ignore", divide="ignore"):
        out = num / (den[..., None] if o.ndim == lse.ndim + 1 else den)
        lse_out = Ms + np.log(den)
    if o.ndim == lse.ndim + 1:
        out = np.where(empty[..., None], 0.0, out)
    else:
        out = np.where(empty, 0.0, out)
    lse_out = np.where(empty, -np.inf, lse_out)
    return out, lse_out
