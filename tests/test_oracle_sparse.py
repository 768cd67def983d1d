"""Pins for the sparse (selected-token) attention oracle (oracle/sparse.py):
dense attention when every token is selected, torch's scaled_dot_product_attention
with the selection as its mask, set semantics (order, duplicates, unused and
invisible entries), closed forms, relocation and poisoning.  CPU only."""
from dataclasses import replace

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import sparse as OS
from paged_attention_quantized_gb300 import workloads as W
from tests.oracle_ref import decode_rows

CASES = [
    ("tiny", dict()),
    ("bf16", dict(B=3, L_lo=5, L_hi=90, Hq=8, Hkv=2, n=2)),
    ("e4m3", dict(B=2, L_lo=5, L_hi=90, Hq=4, Hkv=2, n=4)),
    ("int8", dict(B=2, L_lo=10, L_hi=60, Hq=4, Hkv=2)),
    ("int4", dict(B=2, L_lo=10, L_hi=60, Hq=4, Hkv=2)),
    ("latent", dict(B=2, L_lo=5, L_hi=150, Hq=4)),
]


def _soft(w):
    if w.kv_dtype in ("int8", "int4"):
        w.q = (w.q.float() / 3e4).to(w.q.dtype)   # a softmax that mixes tokens
    return w


@pytest.mark.parametrize("name,kw", CASES, ids=lambda x: str(x))
def test_selecting_every_token_is_dense_attention_bitwise(name, kw):
    w = _soft(W.make(name, **kw))
    L = w.context_lens.tolist()
    k = max(L) + 5
    sel = torch.full((w.B, w.n, k), -1, dtype=torch.int32)
    g = torch.Generator().manual_seed(1)
    for b, Lb in enumerate(L):
        for j in range(w.n):
            sel[b, j, :Lb] = torch.randperm(Lb, generator=g).to(torch.int32)   # includes invisible ones
    out, lse = OS.sparse_attention(w, sel)
    ref, rlse = oracle.attention(w, threads=2)
    assert np.array_equal(out, ref) and np.array_equal(lse, rlse)


@pytest.mark.parametrize("name,kw", CASES, ids=lambda x: str(x))
def test_matches_sdpa_with_selection_mask(name, kw):
    w = _soft(W.make(name, **kw))
    sel = W.make_selection(w, k=17, seed=3, shared=0.7)
    out, lse = OS.sparse_attention(w, sel)
    out = out.reshape(w.B, w.n, w.Hq, w.Dv)
    lse = lse.reshape(w.B, w.n, w.Hq)
    K = decode_rows(w, w.k_pool, w.Dk, "k")
    V = decode_rows(w, w.k_pool if w.v_is_k_prefix else w.v_pool, w.Dv, "v")
    tab = w.block_table.to(torch.int64)
    G = w.Hq // w.Hkv
    for b, Lb in enumerate(w.context_lens.tolist()):
        t = torch.arange(Lb)
        Kb = K[tab[b, t // w.bs], :, t % w.bs].permute(1, 0, 2).repeat_interleave(G, 0)   # [Hq, L, Dk]
        Vb = V[tab[b, t // w.bs], :, t % w.bs].permute(1, 0, 2).repeat_interleave(G, 0)
        for j in range(w.n):
            vis = Lb - (w.n - 1 - j) if w.causal else Lb
            mask = torch.zeros(Lb, dtype=torch.bool)
            s = sel[b, j].to(torch.int64)
            s = s[(s >= 0) & (s < vis)]
            mask[s] = True
            qh = w.q[b, j].double()[:, None, :]          # [Hq, 1, Dk]
            if not mask.any():
                assert np.all(out[b, j] == 0) and np.all(np.isneginf(lse[b, j]))
                continue
            o = F.scaled_dot_product_attention(qh, Kb, Vb, attn_mask=mask[None, None, :],
                                               scale=w.softmax_scale)[:, 0]
            sc = (qh @ Kb.transpose(1, 2))[:, 0] * w.softmax_scale
            ls = torch.logsumexp(sc.masked_fill(~mask[None], -float("inf")), dim=-1)
            scale = max(1.0, float(o.abs().max()))
            assert np.max(np.abs(out[b, j] - o.numpy())) <= 1e-12 * scale
            assert np.max(np.abs(lse[b, j] - ls.numpy())) <= 1e-10 * max(1.0, float(ls.abs().max()))


def test_order_duplicates_unused_and_invisible_entries_do_not_matter():
    w = W.make("e4m3", B=2, L_lo=30, L_hi=90, Hq=4, Hkv=2, n=3)
    sel = W.make_selection(w, k=12, seed=4)
    out, lse = OS.sparse_attention(w, sel)
    g = torch.Generator().manual_seed(9)
    L = w.context_lens.tolist()
    extra = torch.full((w.B, w.n, 20), -1, dtype=torch.int32)
    for b in range(w.B):
        for j in range(w.n):
            vis = L[b] - (w.n - 1 - j)
            row = sel[b, j][torch.randperm(12, generator=g)]
            dup = row[:5]                                         # listed twice
            invisible = torch.arange(vis, vis + 3, dtype=torch.int32)  # at or past the visible length
            extra[b, j, :20] = torch.cat([row, dup, invisible])
    out2, lse2 = OS.sparse_attention(w, extra)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_empty_and_single_token_selections():
    w = W.make("bf16", B=2, L_lo=20, L_hi=40, Hq=4, Hkv=2)
    sel = torch.full((w.B, 1, 4), -1, dtype=torch.int32)
    sel[1, 0, 2] = 7
    out, lse = OS.sparse_attention(w, sel)
    out = out.reshape(w.B, 1, w.Hq, w.Dv)
    lse = lse.reshape(w.B, 1, w.Hq)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    V = decode_rows(w, w.v_pool, w.Dv, "v")
    K = decode_rows(w, w.k_pool, w.Dk, "k")
    blk, slot = int(w.block_table[1, 7 // w.bs]), 7 % w.bs
    for h in range(w.Hq):
        g = h // (w.Hq // w.Hkv)
        assert np.array_equal(out[1, 0, h], V[blk, g, slot].numpy())
        s = float(w.q[1, 0, h].double() @ K[blk, g, slot]) * w.softmax_scale
        assert abs(lse[1, 0, h] - s) <= 1e-12 * max(1.0, abs(s))


@pytest.mark.parametrize("name", ["bf16", "int4", "latent"])
def test_relocation_invariance_bitwise(name):
    w = W.make(name, B=2, L_lo=20, L_hi=120, Hq=4, Hkv=1 if name == "latent" else 2, n=2)
    sel = W.make_selection(w, k=16, seed=5)
    out, lse = OS.sparse_attention(w, sel)
    o2, l2 = OS.sparse_attention(W.relocate(w, seed=3), sel)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)


def test_unselected_tokens_never_reach_the_output():
    # every byte of every token no row selects becomes an E4M3 NaN code
    w = W.make("e4m3", B=2, L_lo=40, L_hi=90, Hq=4, Hkv=2, n=2, poison=False)
    sel = W.make_selection(w, k=10, seed=6)
    out, lse = OS.sparse_attention(w, sel)
    kp, vp = w.k_pool.clone(), w.v_pool.clone()
    row = w.k_row_bytes
    L = w.context_lens.tolist()
    for b, Lb in enumerate(L):
        used = set()
        for j in range(w.n):
            used |= set(OS.selected(sel[b, j].numpy(), Lb - (w.n - 1 - j)).tolist())
        for t in range(Lb):
            if t in used:
                continue
            blk, slot = int(w.block_table[b, t // w.bs]), t % w.bs
            for g in range(w.Hkv):
                o = (g * w.bs + slot) * row
                kp[blk, o:o + row] = 0x7F
                vp[blk, o:o + row] = 0xFF
    o2, l2 = OS.sparse_attention(replace(w, k_pool=kp, v_pool=vp), sel)
    assert np.isfinite(o2).all()
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)


def test_selection_recipe():
    w = W.make("bf16", B=3, L_lo=200, L_hi=400, Hq=4, Hkv=2, n=3)
    w.causal = True
    sel = W.make_selection(w, k=64, seed=7, shared=0.9)
    assert sel.shape == (3, 3, 64) and sel.dtype == torch.int32
    L = w.context_lens.tolist()
    for b in range(3):
        for j in range(3):
            s = sel[b, j]
            assert ((s >= 0) & (s < L[b] - (2 - j))).all()
        # rows of one request share most of their selection
        a, c = set(sel[b, 0].tolist()), set(sel[b, 2].tolist())
        assert len(a & c) >= 0.7 * 64
    short = W.make("bf16", context_lens=[5, 70], Hq=4, Hkv=2)
    s2 = W.make_selection(short, k=8, seed=1)
    assert sorted(s2[0, 0, :5].tolist()) == [0, 1, 2, 3, 4] and (s2[0, 0, 5:] == -1).all()
