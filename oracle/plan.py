"""Work plan definition -- TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The rule the device planner must follow, written plainly so that its output
can be compared element by element.  It is a function of the context lengths
and fixed sizes only; block ids never enter it, so the work order -- and with
it every reduction order -- cannot depend on where the allocator put a page
(1Cat-vLLM PR #494, "[Bugfix][SM70] Stabilize QSA page4 order under KV
relocation", Summary: order by logical position, physical addresses are only
payload).

Rule
----
  P_b  = ceil(L_b / bs) pages of request b; a request with L_b < 0,
         L_b > max_context_len or P_b > max_blocks_per_seq is invalid:
         flagged, and planned with P_b = 0.
  W    = sum_b P_b
  T    = max(1, target_ctas // (Hkv * row_blocks))
  C    = forced_pages if forced_pages > 0 else max(min_pages, ceil(W / T))
  S_b  = max(1, ceil(P_b / C))          (splits of request b)
  ofs_b = sum_{b' < b} S_b'
  unit index  u = ofs_b * Hkv + h * S_b + s   for kv head h, split s
  unit pages  [s * C, min((s + 1) * C, P_b))
"""
from __future__ import annotations

import numpy as np


def plan(context_lens, *, bs: int, Hkv: int, max_context_len: int, max_blocks_per_seq: int,
         target_ctas: int, min_pages: int, row_blocks: int = 1, forced_pages: int = 0):
    L = np.asarray(context_lens, dtype=np.int64).reshape(-1)
    B = L.size
    P = np.zeros(B, dtype=np.int64)
    flags = np.zeros(B, dtype=np.int64)
    for b in range(B):
        pb = -(-L[b] // bs) if L[b] > 0 else 0
        if L[b] < 0 or L[b] > max_context_len or pb > max_blocks_per_seq:
            flags[b] = 1
            pb = 0
        P[b] = pb
    W = int(P.sum())
    T = max(1, target_ctas // (Hkv * row_blocks))
    if forced_pages > 0:
        C = forced_pages
    else:
        C = max(min_pages, -(-W // T))
    S = np.maximum(1, -(-P // C))
    ofs = np.concatenate([[0], np.cumsum(S)[:-1]]) if B else np.zeros(0, dtype=np.int64)
    units = []
    for b in range(B):
        for h in range(Hkv):
            for s in range(S[b]):
                units.append((b, h, s, min(s * C, P[b]), min((s + 1) * C, P[b])))
    return {
        "chunk_pages": C,
        "splits": S.astype(np.int64),
        "offsets": ofs.astype(np.int64),
        "flags": flags,
        "pages": P,
        "num_units": int(S.sum()) * Hkv,
        "units": units,   # in unit-index order
    }
