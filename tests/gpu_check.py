"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle on the same bytes."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import paged_attention_quantized_gb300 as pa

# max-abs tolerances on the output (fp32 output 2e-3, bf16 / fp16 output 1e-2);
# fp32 outputs of per-channel INT8/INT4 caches (magnitudes up to 1e5) are
# compared normwise, see compare()
TOL = {"f32": 2e-3, "bf16": 1e-2, "f16": 1e-2}
MAX_CODE = {"int8": 127.0, "int4": 7.0}


def run_gpu(w, *, steps="all", **pkw):
    p = pa.problem(w, **pkw)
    out, lse, ws = pa.alloc(w, p)
    pa.run(w, p, out, ws, lse, steps=steps)
    torch.cuda.synchronize()
    return out, lse, ws, p


def error_bits(ws) -> int:
    return pa.binding().pa_get_error(ws.data_ptr(), pa.stream_handle())


def sample_rows(w, count: int, seed: int = 0) -> np.ndarray:
    """Seeded (b, j, h) rows, always including every row of the longest request's
    first and last query head."""
    rng = np.random.default_rng(seed)
    L = w.context_lens.cpu().numpy()
    bmax = int(np.argmax(L))
    rows = {(bmax, j, h) for j in range(w.n) for h in (0, w.Hq - 1)}
    while len(rows) < count:
        rows.add((int(rng.integers(w.B)), int(rng.integers(w.n)), int(rng.integers(w.Hq))))
    return np.array(sorted(rows), dtype=np.int64)


def fold_eps(w, rows) -> np.ndarray:
    """First-order bound on |GPU score - exact score| for per-channel INT8/INT4
    rows: the fold rounds q * k_scale / max|k_scale| once to f16 (relative
    2^-11, doubled for margin), times softmax_scale * max|code| * sum_d
    |q_d| k_scale_d."""
    q = w.q.detach().cpu().to(torch.float64).numpy()
    ks = w.k_scale.detach().cpu().to(torch.float64).numpy()
    G = w.Hq // w.Hkv
    out = np.zeros(len(rows))
    for i, (b, j, h) in enumerate(rows):
        out[i] = 2.0 ** -10 * w.softmax_scale * MAX_CODE[w.kv_dtype] * float(np.sum(np.abs(q[b, j, h]) * ks[h // G]))
    return out


def hull_delta(w, rows, eps, tol) -> np.ndarray:
    """Score window of the near-tie check, per row.

    Every GPU score is within eps of the exact one, so the GPU's softmax
    weight of a token scoring d below the exact maximum is at most
    exp(-(d - 2 eps)) times that of the maximal token.  With
    delta = 2 eps + ln(2 (vis - 1) Vmax / tol), the tokens outside the window
    together weigh at most tol / (2 Vmax), so they move any output channel by
    at most tol (values differ by at most 2 Vmax), and the GPU output is a
    convex combination of the window's values up to that tol.  Vmax is
    bounded by max|code| * max_d |v_scale[g, d]|."""
    L = w.context_lens.cpu().numpy().astype(np.int64)
    vs = np.abs(w.v_scale.detach().cpu().to(torch.float64).numpy())
    G = w.Hq // w.Hkv
    out = np.zeros(len(rows))
    for i, (b, j, h) in enumerate(rows):
        vis = int(L[b]) - (w.n - 1 - int(j)) if w.causal else int(L[b])
        vmax = MAX_CODE[w.kv_dtype] * float(vs[int(h) // G].max())
        out[i] = 2.0 * eps[i] + math.log(max(1.0, 2.0 * max(vis - 1, 0) * vmax / tol))
    return out


def abs_values(w):
    """The workload with every V code replaced by its absolute value: its exact
    output is sum_t p_t |v_t|, the magnitude scale of each output element."""
    import dataclasses
    v = w.v_pool
    if w.kv_dtype == "int8":
        nv = v.view(torch.int8).abs().view(torch.uint8)
    elif w.kv_dtype == "int4":
        lo = ((v.to(torch.int16) << 12) >> 12).abs()      # sign-extended low nibble
        hi = ((v.to(torch.int16) << 8) >> 12).abs()
        nv = ((lo & 0xF) | ((hi & 0xF) << 4)).to(torch.uint8)
    else:
        raise ValueError(w.kv_dtype)
    vs = None if w.v_scale is None else w.v_scale.abs()
    return dataclasses.replace(w, v_pool=nv.contiguous(), v_scale=vs)


def compare(w, out, lse, rows=None, host=None, report=None, ref=None):
    """Assert GPU rows match the oracle.  Returns (max_err, n_hull_rows).

    fp16 / bf16 / fp32 outputs use the absolute tolerances above.  Per-channel
    INT8 / INT4 outputs (magnitudes up to 1e5, heavy cancellation between
    tokens) are compared normwise: |gpu - ref| <= tol * max(1, sum_t p_t |v_t|).
    Where the fold's score error (fold_eps) can move softmax weights by more
    than tol, a row that misses this may still pass if it lies, per channel,
    inside the values of the tokens whose exact score is within hull_delta of
    the maximum (the near-tie rule of the onnxruntime PR #32520 page,
    Validation status: the argmax of a near one-hot softmax depends on fp16
    rounding).  `report` (a dict) receives the largest error and the number
    of rows accepted through the hull.  `ref` = (out, lse) of the oracle on
    `rows`, when the caller has evaluated them already."""
    if rows is None:
        grid = np.stack(np.meshgrid(np.arange(w.B), np.arange(w.n), np.arange(w.Hq), indexing="ij"), -1)
        rows = grid.reshape(-1, 3)
    rows = np.asarray(rows, dtype=np.int64)
    host = host or oracle.HostArrays(w)
    if ref is None:
        ref, rlse = oracle.attention(w, rows=rows, host=host)
    else:
        ref, rlse = ref  # the oracle's rows, already evaluated by the caller
    o = out.detach().float().cpu().numpy().astype(np.float64)
    l = lse.detach().float().cpu().numpy().astype(np.float64)
    g = o[rows[:, 0], rows[:, 1], rows[:, 2]]
    gl = l[rows[:, 0], rows[:, 1], rows[:, 2]]
    tol = TOL[w.out_dtype]
    assert np.isfinite(g).all(), "GPU output has non-finite values"
    per_channel_int = w.kv_dtype in ("int8", "int4") and w.k_scale_mode == "channel"
    eps = np.zeros(len(rows))
    if per_channel_int:
        mag, _ = oracle.attention(abs_values(w), rows=rows)
        allow = tol * np.maximum(1.0, mag)
        eps = fold_eps(w, rows)
    else:
        allow = np.full_like(g, tol)
    err = np.abs(g - ref)
    bad = err > allow
    n_hull = 0
    n_ties = 0
    if per_channel_int and bad.any():
        cand = np.nonzero(bad.any(axis=1))[0]
        delta = hull_delta(w, rows[cand], eps[cand], tol)
        for i, dl in zip(cand, delta):
            if 4.0 * eps[i] <= tol:
                continue  # weights cannot move enough: a real failure
            b, j, h = (int(x) for x in rows[i])
            vmin, vmax, gap, cnt = oracle.row_ties(w, b, j, h, float(dl), host=host)
            # the window's values, widened by the tolerance and by the (at
            # most tol) pull of the tokens outside it
            lo = vmin - tol * np.maximum(1.0, np.abs(vmin)) - tol
            hi = vmax + tol * np.maximum(1.0, np.abs(vmax)) + tol
            if np.all((g[i] >= lo) & (g[i] <= hi)):
                bad[i] = False
                n_hull += 1
                n_ties += int(gap < 2.0 * eps[i])
    if bad.any():
        i = np.argwhere(bad)[0]
        r = rows[i[0]]
        raise AssertionError(f"row (b,j,h)={tuple(r)} d={i[1]}: gpu {g[i[0], i[1]]!r} vs oracle "
                             f"{ref[i[0], i[1]]!r} (allowed {allow[i[0], i[1]]})")
    # log-sum-exp: same visibility, close values
    fin = np.isfinite(rlse)
    assert np.array_equal(fin, np.isfinite(gl)), "lse visibility differs"
    lerr = np.abs(gl[fin] - rlse[fin])
    ok = lerr <= 1e-3 * np.maximum(1.0, np.abs(rlse[fin])) + 2.0 * eps[fin]
    assert ok.all(), f"lse mismatch: max err {lerr.max()}"
    if report is not None:
        report["max_err"] = float(err.max(initial=0.0))
        report["hull_rows"] = n_hull
        report["tie_rows"] = n_ties
        report["rows"] = int(len(rows))
    return float(err.max(initial=0.0)), n_hull
