"""CPU oracle for sparse (selected-token) paged attention -- TEST
INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg
may use this module; the product path never does, and nothing here is shared
with it.

What it computes: query row j of request b (every head) attends only to the
logical token positions its selection names, instead of to all of
[0, vis).  For request b, row j, head h (kv head g = h / (Hq / Hkv)):

    T_bj  = { t in sel[b][j][:] : 0 <= t < vis_bj }      (a set)
    out   = softmax_{t in T_bj}( softmax_scale * q[b,j,h,:] . k^_t ) . v^_t
    lse   = ln sum_{t in T_bj} exp(...);   T_bj empty gives out = 0, lse = -inf

with vis_bj = L_b - (next_n - 1 - j) (causal) or L_b, and k^_t, v^_t the
dequantized rows of token t found through block_table exactly as for dense
attention.

Sources (page title, section):
  * 1Cat-vLLM PR #494, "[Bugfix][SM70] Stabilize QSA page4 order under KV
    relocation", Summary / Investigation / Contract and limits: sparse (QSA)
    attention over per-query selected token ids; results depend on the
    logical selections only -- never on physical page ids or on the order in
    which selections are listed -- and are bitwise stable under relocation.
  * the same page, Upstream and duplicate-work check: unused selection
    entries are skipped.

Readings where the pages are silent: one selection per query token, shared
by all its heads; entries < 0 are unused; a selected position at or past
the row's visible length is skipped like an unused entry (causality still
holds); a position listed twice counts once (a selection is a set).

How: the selected tokens' code rows (and per-token scales) are copied, in
ascending logical order, into a compacted pool of one-token blocks, and the
dense oracle (`oracle.attention`, which walks tokens in logical order) runs
on it -- the definition above is dense attention over the selected set.
Byte copies only; all arithmetic is the dense oracle's.

Functions
---------
selected(sel_row, vis) -> sorted unique visible positions
sparse_attention(w, sel, rows=None) -> (out [rows, Dv] float64, lse [rows])
"""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import torch

from . import attention

_BITS = {"f16": 16, "bf16": 16, "e4m3": 8, "int8": 8, "int4": 4}


def selected(sel_row, vis: int) -> np.ndarray:
    """The set a selection row names: entries in [0, vis), ascending, once each."""
    s = np.asarray(sel_row, dtype=np.int64).reshape(-1)
    return np.unique(s[(s >= 0) & (s < vis)])


def _host(t):
    return t.detach().cpu() if hasattr(t, "detach") else torch.as_tensor(t)


def _compact(w, b: int, toks: np.ndarray):
    """A one-request workload whose logical tokens 0..m-1 are tokens `toks` of
    request b (one token per block, block i+1 holds toks[i]); the null block 0
    is all zero bytes."""
    m = len(toks)
    bits = _BITS[w.kv_dtype]
    table = _host(w.block_table).numpy()
    blk = table[b, toks // w.bs] if m else np.zeros(0, np.int64)
    slot = toks % w.bs

    def plane(pool, D, tok_scaled):
        if pool is None:
            return None
        src = _host(pool).numpy()
        row = D * bits // 8
        codes = w.Hkv * w.bs * row
        out_bb = w.Hkv * row + (w.Hkv * 4 if tok_scaled else 0)
        out = np.zeros((m + 1, out_bb), dtype=np.uint8)
        for g in range(w.Hkv):
            o = (g * w.bs + slot) * row
            idx = o[:, None] + np.arange(row)[None, :]
            out[1:, g * row:(g + 1) * row] = src[blk[:, None], idx]
            if tok_scaled:
                so = codes + (g * w.bs + slot) * 4
                sidx = so[:, None] + np.arange(4)[None, :]
                out[1:, w.Hkv * row + g * 4: w.Hkv * row + (g + 1) * 4] = src[blk[:, None], sidx]
        return torch.from_numpy(out)

    k_tok = w.k_scale_mode == "token"
    v_tok = w.v_scale_mode == "token"
    kp = plane(w.k_pool, w.Dk, k_tok)
    vp = None if w.v_is_k_prefix else plane(w.v_pool, w.Dv, v_tok)
    tab = torch.arange(1, m + 1, dtype=torch.int32).reshape(1, max(m, 0))
    if m == 0:
        tab = torch.zeros((1, 1), dtype=torch.int32)
    return replace(w, B=1, n=1, bs=1, num_blocks=m + 1, max_blocks_per_seq=max(1, m),
                   max_context_len=max(1, m), causal=False, k_pool=kp, v_pool=vp,
                   block_table=tab, context_lens=torch.tensor([m], dtype=torch.int32),
                   k_scale=None if w.k_scale is None else _host(w.k_scale),
                   v_scale=None if w.v_scale is None else _host(w.v_scale))


def sparse_attention(w, sel, rows=None):
    """Sparse attention for the given (b, j, h) rows (default: all, in (b, j, h)
    order).  sel: [B, next_n, K] int32 selected logical positions per query
    token.  Returns (out [num_rows, Dv] float64, lse [num_rows] float64)."""
    sel = _host(sel).numpy() if hasattr(sel, "detach") else np.asarray(sel)
    lens = _host(w.context_lens).numpy()
    q = _host(w.q)
    if rows is None:
        grid = np.stack(np.meshgrid(np.arange(w.B), np.arange(w.n), np.arange(w.Hq), indexing="ij"), -1)
        rows = grid.reshape(-1, 3)
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
    out = np.zeros((len(rows), w.Dv), dtype=np.float64)
    lse = np.zeros(len(rows), dtype=np.float64)
    # one compacted workload per (b, j): every head of that query token
    order = {}
    for i, (b, j, h) in enumerate(rows):
        order.setdefault((int(b), int(j)), []).append((i, int(h)))
    for (b, j), items in order.items():
        vis = int(lens[b]) - (w.n - 1 - j) if w.causal else int(lens[b])
        toks = selected(sel[b, j], vis)
        wc = _compact(w, b, toks)
        wc = replace(wc, q=q[b:b + 1, j:j + 1].contiguous())
        o, l = attention(wc, rows=[(0, 0, h) for _, h in items], threads=1)
        for k, (i, _) in enumerate(items):
            out[i] = o[k]
            lse[i] = l[k]
    return out, lse
