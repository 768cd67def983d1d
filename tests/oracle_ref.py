"""Independent routes to the oracle's quantities, used only to pin the oracle.

Nothing here re-types the oracle's formulas: codes are decoded through library
conversions (torch's float16 / bfloat16 / float8_e4m3fn views, numpy's int8
view and arithmetic shifts), tokens are gathered with tensor indexing, and the
attention itself is torch's scaled_dot_product_attention in float64.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


def decode_rows(w, pool: torch.Tensor, D: int, which: str) -> torch.Tensor:
    """float64 [num_blocks, Hkv, bs, D] values (code * scale) of a pool plane."""
    pool = pool.cpu()
    nb = pool.shape[0]
    bits = {"f16": 16, "bf16": 16, "e4m3": 8, "int8": 8, "int4": 4}[w.kv_dtype]
    row_bytes = D * bits // 8
    plane_row = (w.Dk * bits // 8) if (which == "v" and w.v_is_k_prefix) else row_bytes
    codes_bytes = w.Hkv * w.bs * plane_row
    raw = pool[:, :codes_bytes].reshape(nb, w.Hkv, w.bs, plane_row)[..., :row_bytes].contiguous()
    if w.kv_dtype == "f16":
        vals = raw.view(torch.float16).to(torch.float64)
    elif w.kv_dtype == "bf16":
        vals = raw.view(torch.bfloat16).to(torch.float64)
    elif w.kv_dtype == "e4m3":
        vals = raw.view(torch.float8_e4m3fn).to(torch.float64)
    elif w.kv_dtype == "int8":
        vals = raw.view(torch.int8).to(torch.float64)
    else:
        b = raw.numpy()
        lo = (b.astype(np.uint8) << 4).astype(np.int8) >> 4
        hi = b.astype(np.int8) >> 4
        v = np.empty(b.shape[:-1] + (b.shape[-1] * 2,), dtype=np.float64)
        v[..., 0::2] = lo
        v[..., 1::2] = hi
        vals = torch.from_numpy(v)
    mode = w.k_scale_mode if (which == "k" or w.v_is_k_prefix) else w.v_scale_mode
    scale = w.k_scale if (which == "k" or w.v_is_k_prefix) else w.v_scale
    if mode == "tensor":
        vals = vals * float(scale.cpu()[0])
    elif mode == "channel":
        full_D = w.Dk if (which == "k" or w.v_is_k_prefix) else w.Dv
        vals = vals * scale.cpu().to(torch.float64).reshape(1, w.Hkv, 1, full_D)[..., :D]
    elif mode == "token":
        tail = pool[:, codes_bytes: codes_bytes + w.Hkv * w.bs * 4].contiguous()
        vals = vals * tail.view(torch.float32).to(torch.float64).reshape(nb, w.Hkv, w.bs, 1)
    return vals


def reference(w):
    """(out [B, n, Hq, Dv] float64, lse [B, n, Hq]) by SDPA over gathered tokens."""
    K = decode_rows(w, w.k_pool, w.Dk, "k")
    V = decode_rows(w, w.k_pool if w.v_is_k_prefix else w.v_pool, w.Dv, "v")
    q = w.q.cpu().to(torch.float64)
    table = w.block_table.cpu().to(torch.int64)
    lens = w.context_lens.cpu().tolist()
    G = w.Hq // w.Hkv
    out = torch.zeros((w.B, w.n, w.Hq, w.Dv), dtype=torch.float64)
    lse = torch.full((w.B, w.n, w.Hq), -float("inf"), dtype=torch.float64)
    for b, L in enumerate(lens):
        if L <= 0:
            continue
        t = torch.arange(L)
        blk = table[b, t // w.bs]
        slot = t % w.bs
        Kb = K[blk, :, slot]            # [L, Hkv, Dk]
        Vb = V[blk, :, slot]            # [L, Hkv, Dv]
        Kh = Kb.permute(1, 0, 2).repeat_interleave(G, dim=0)   # [Hq, L, Dk]
        Vh = Vb.permute(1, 0, 2).repeat_interleave(G, dim=0)
        qb = q[b].permute(1, 0, 2)     # [Hq, n, Dk]
        pos = L - w.n + torch.arange(w.n) if w.causal else torch.full((w.n,), L - 1)
        mask = t[None, :] <= pos[:, None]  # [n, L]
        ok = mask.any(dim=1)
        o = F.scaled_dot_product_attention(qb[None], Kh[None], Vh[None],
                                           attn_mask=mask[None, None], scale=w.softmax_scale)[0]
        s = torch.matmul(qb, Kh.transpose(1, 2)) * w.softmax_scale
        s = s.masked_fill(~mask[None], -float("inf"))
        ls = torch.logsumexp(s, dim=-1)   # [Hq, n]
        o = torch.where(ok[None, :, None], o, torch.zeros_like(o))
        out[b] = o.permute(1, 0, 2)
        lse[b] = torch.where(ok[None, :], ls, torch.full_like(ls, -float("inf"))).permute(1, 0)
    return out.numpy(), lse.numpy()
