"""Work plan definition -- TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The rule the device planner and the attention launch must follow, written
plainly so that their records can be compared element by element.  It is a
function of the context lengths and fixed sizes only; block ids never enter
it, so the work order -- and with it every reduction order -- cannot depend on
where the allocator put a page (1Cat-vLLM PR #494, "[Bugfix][SM70] Stabilize
QSA page4 order under KV relocation", Summary: order by logical position,
physical addresses are only payload).

Rule
----
  P_b   = ceil(L_b / bs) pages of request b (bs: tokens of a work page); a
          request with L_b < 0, L_b > max_context_len or more blocks of
          block_size tokens (default bs) than max_blocks_per_seq is invalid:
          flagged, and planned with P_b = 0.
  PS_b  = sum_{b' < b} P_b'                       (request record)
  X     = Hkv * row_blocks                        (segments per request)
  segment s = b * X + q covers positions PS_b * X + q * P_b + [0, P_b)
  N     = X * sum_b P_b positions in all
  warp k of W takes positions [k N / W, (k + 1) N / W)   (integer division)
  piece = a warp's positions inside one segment; its partial slot is s + k;
  a piece that is a whole segment is "complete" (written as the output).

Grouped workers (group_size G > 1, the single-latent kernel: one worker per
row block of a kv head): positions run over (request, kv head, page) only --
U = X / G units per request, unit u = segments u*G .. u*G + G-1 --, the
W / G worker groups share them as above, and worker g*G + i of group g takes
row block i of every unit in the group's share.  The piece of segment
s = b*X + u*G + i in group g has partial slot (b*U + u + g)*G + i; slots in
all: (B*U + W/G)*G.  G = 1 is the rule above.
"""
from __future__ import annotations

import numpy as np


def plan(context_lens, *, bs: int, Hkv: int, max_context_len: int, max_blocks_per_seq: int,
         row_blocks: int = 1, warps: int = 1, group_size: int = 1, block_size: int | None = None):
    L = np.asarray(context_lens, dtype=np.int64).reshape(-1)
    B = L.size
    P = np.zeros(B, dtype=np.int64)
    flags = np.zeros(B, dtype=np.int64)
    tb = bs if block_size is None else block_size
    for b in range(B):
        pb = -(-L[b] // bs) if L[b] > 0 else 0
        nblocks = -(-L[b] // tb) if L[b] > 0 else 0
        if L[b] < 0 or L[b] > max_context_len or nblocks > max_blocks_per_seq:
            flags[b] = 1
            pb = 0
        P[b] = pb
    PS = np.concatenate([[0], np.cumsum(P)[:-1]]).astype(np.int64) if B else np.zeros(0, dtype=np.int64)
    X = Hkv * row_blocks
    G = group_size
    assert X % G == 0 and warps % G == 0
    U = X // G
    NG = warps // G
    N = int(P.sum()) * U
    starts = [g * N // NG for g in range(NG + 1)]
    pieces = []
    for b in range(B):
        for u in range(U):
            if P[b] == 0:
                continue
            o0 = int(PS[b]) * U + u * int(P[b])
            o1 = o0 + int(P[b])
            for g in range(NG):
                lo, hi = max(o0, starts[g]), min(o1, starts[g + 1])
                if lo < hi:
                    for i in range(G):
                        s = b * X + u * G + i
                        pieces.append({"segment": s, "warp": g * G + i, "slot": (b * U + u + g) * G + i,
                                       "pages": (lo - o0, hi - o0), "complete": lo == o0 and hi == o1})
    return {"pages": P, "prefix": PS, "flags": flags, "total_pages": int(P.sum()), "positions": N,
            "warp_starts": starts, "pieces": pieces, "slots": (B * U + NG) * G}
