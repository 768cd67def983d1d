"""Pins for the FP4 (MXFP4) paged MQA logits oracle: format values, the
page's worked precondition and interleave formula, brute force on tiny
inputs, closed forms and invariances.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import mqa_logits as M
from paged_attention_quantized_gb300 import workloads as W

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "fp4_formats.json")))


def test_e2m1_values_are_the_format_table():
    want = np.array(GOLDEN["e2m1_values"]["codes_0_to_15"])
    got = M.e2m1_table()
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))      # code 8 is -0


def test_ue8m0_matches_torch_e8m0():
    b = torch.arange(256, dtype=torch.int16).to(torch.uint8)
    ref = b.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = M.ue8m0_table()
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127


def test_table_precondition_worked_case():
    g = GOLDEN["table_columns"]
    assert M.required_table_columns(g["context_len"], g["block_size"]) == g["columns"]
    assert M.required_table_columns(256, 64) == 4 and M.required_table_columns(1, 16) == 8


def test_interleaved_scale_slots():
    g = GOLDEN["interleaved_scales"]
    bs = g["block_size"]
    assert [M.sf_slot_token(k, bs, True) for k in range(8)] == g["tokens_of_slots_0_to_7"]
    for bs in (4, 16, 64, 128):
        assert sorted(M.sf_slot_token(k, bs, True) for k in range(bs)) == list(range(bs))
        assert [M.sf_slot_token(k, bs, False) for k in range(bs)] == list(range(bs))


def _brute(w, r):
    """Logits of row r by explicit loops over heads, channels and tokens,
    decoding with the format table above and torch's E8M0."""
    e2m1 = GOLDEN["e2m1_values"]["codes_0_to_15"]
    e8 = torch.arange(256, dtype=torch.int16).to(torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).tolist()
    b, j = divmod(r, w.n)
    L = int(w.context_lens[b])
    vis = L - (w.n - 1 - j) if w.causal else L
    q = w.q.numpy()
    sfq = w.sf_q.numpy().astype(np.int64) & 0xFFFFFFFF
    kv = w.kv_fused.numpy()
    half = w.D // 2
    out = [-math.inf] * w.max_context_len
    for t in range(max(vis, 0)):
        blk = int(w.block_table[b, t // w.bs])
        slot = t % w.bs
        ws = slot
        if w.sf_interleaved:
            ws = [k for k in range(w.bs) if (k % 4) * (w.bs // 4) + k // 4 == slot][0]
        acc = 0.0
        for h in range(w.H):
            dot = 0.0
            for d in range(w.D):
                qb = int(q[b, j, h, d // 2])
                qc = (qb >> 4) if d % 2 else (qb & 15)
                qs = e8[(int(sfq[b, j, h]) >> (8 * (d // 32))) & 0xFF]
                kb = int(kv[blk, slot * half + d // 2])
                kc = (kb >> 4) if d % 2 else (kb & 15)
                ks = e8[int(kv[blk, w.bs * half + ws * 4 + d // 32])]
                dot += e2m1[qc] * qs * e2m1[kc] * ks
            if w.rectify:
                dot = max(dot, 0.0)
            acc += float(w.weights[r, h]) * dot
        out[t] = acc
    return np.array(out)


@pytest.mark.parametrize("kw", [dict(), dict(causal=False), dict(rectify=True), dict(sf_interleaved=True, bs=16)])
def test_brute_force_tiny(kw):
    base = dict(B=2, n=2, H=3, bs=32, context_lens=[5, 40], scale_lo=120, scale_hi=134)
    base.update(kw)
    w = W.make_fp4(**base)
    out = M.mqa_logits(w)
    for r in range(w.B * w.n):
        ref = _brute(w, r)
        fin = np.isfinite(ref)
        assert np.array_equal(fin, np.isfinite(out[r]))
        assert np.allclose(out[r][fin], ref[fin], rtol=1e-12, atol=1e-9)
        assert np.all(np.isneginf(out[r][~fin]))


def _small(**kw):
    base = dict(B=3, n=2, H=8, bs=64, L_lo=50, L_hi=400)
    base.update(kw)
    return W.make_fp4(**base)


def test_zero_k_codes_give_zero_logits():
    w = _small()
    kv = w.kv_fused.clone()
    data = w.bs * (w.D // 2)
    kv[:, :data] = 0
    w.kv_fused = kv
    out = M.mqa_logits(w)
    L = w.context_lens.numpy()
    for r in range(w.B * w.n):
        b, j = divmod(r, w.n)
        vis = L[b] - (w.n - 1 - j)
        assert np.all(out[r, :vis] == 0.0) and np.all(np.isneginf(out[r, vis:]))


def test_scale_bytes_plus_one_double_the_logits():
    w = _small()
    out = M.mqa_logits(w)
    kv = w.kv_fused.clone()
    data = w.bs * (w.D // 2)
    kv[:, data:] = kv[:, data:] + 1         # every in-range scale byte (the junk ones too)
    ref_blocks = set(int(x) for x in w.block_table.reshape(-1))
    w2 = W.Fp4Logits(**{**w.__dict__, "kv_fused": kv})
    out2 = M.mqa_logits(w2)
    fin = np.isfinite(out)
    assert np.array_equal(out2[fin], 2.0 * out[fin])
    sfq = w.sf_q.numpy().astype(np.int64) + 0x01010101   # every q scale byte + 1 as well
    w3 = W.Fp4Logits(**{**w2.__dict__, "sf_q": torch.from_numpy(sfq.astype(np.uint32).view(np.int32))})
    assert np.array_equal(M.mqa_logits(w3)[fin], 4.0 * out[fin])
    assert ref_blocks


def test_weights_are_linear_and_rectify_clamps_each_head():
    w = _small(H=4)
    out = M.mqa_logits(w)
    w2 = W.Fp4Logits(**{**w.__dict__, "weights": w.weights * 2})
    fin = np.isfinite(out)
    assert np.array_equal(M.mqa_logits(w2)[fin], 2.0 * out[fin])
    # one head at a time: the plain logits are w_h * dot_h, the rectified max(0, .)
    parts = []
    for h in range(w.H):
        wh = torch.zeros_like(w.weights)
        wh[:, h] = 1.0
        parts.append(M.mqa_logits(W.Fp4Logits(**{**w.__dict__, "weights": wh})))
    wt = w.weights.numpy().astype(np.float64)
    summed = sum(wt[:, h:h + 1] * np.where(fin, parts[h], 0.0) for h in range(w.H))
    assert np.allclose(out[fin], summed[fin], rtol=1e-12, atol=1e-9)
    wr = W.Fp4Logits(**{**w.__dict__, "rectify": True})
    rect = sum(wt[:, h:h + 1] * np.where(fin, np.maximum(parts[h], 0.0), 0.0) for h in range(w.H))
    assert np.allclose(M.mqa_logits(wr)[fin], rect[fin], rtol=1e-12, atol=1e-9)


def test_relocation_bitwise():
    w = _small()
    out = M.mqa_logits(w)
    assert np.array_equal(M.mqa_logits(W.relocate_fp4(w, seed=3)), out)


def test_interleaved_pool_equals_token_order_pool():
    a = _small(bs=64, sf_interleaved=False)
    b = _small(bs=64, sf_interleaved=True)
    # same seed, same codes; only the scale words sit in other slots
    assert torch.equal(a.q, b.q) and torch.equal(a.block_table, b.block_table)
    assert np.array_equal(M.mqa_logits(a), M.mqa_logits(b))


def test_causal_row_equals_shorter_single_row():
    w = _small(n=3)
    out = M.mqa_logits(w)
    L = w.context_lens.tolist()
    for b in range(w.B):
        for j in range(w.n):
            one = W.Fp4Logits(**{**w.__dict__, "B": 1, "n": 1, "causal": False,
                                 "q": w.q[b:b + 1, j:j + 1], "sf_q": w.sf_q[b:b + 1, j:j + 1],
                                 "weights": w.weights[b * w.n + j: b * w.n + j + 1],
                                 "block_table": w.block_table[b:b + 1],
                                 "context_lens": torch.tensor([L[b] - (w.n - 1 - j)], dtype=torch.int32)})
            assert np.array_equal(M.mqa_logits(one)[0], out[b * w.n + j])


def test_unreferenced_bytes_never_matter_and_nan_scale_is_local():
    w = _small()
    out = M.mqa_logits(w)
    kv = w.kv_fused.clone()
    used = np.zeros(w.num_blocks, dtype=bool)
    for b, L in enumerate(w.context_lens.tolist()):
        used[w.block_table[b, :(L + w.bs - 1) // w.bs].numpy()] = True
    kv[torch.from_numpy(~used)] = 0xFF           # NaN scales and -6 codes everywhere unused
    assert np.array_equal(M.mqa_logits(W.Fp4Logits(**{**w.__dict__, "kv_fused": kv})), out)
    # a NaN scale byte on one visible token poisons that token's logits only
    blk = int(w.block_table[0, 0])
    kv = w.kv_fused.clone()
    kv[blk, w.bs * (w.D // 2) + 3 * 4 + 1] = 0xFF   # token 3, second scale group
    o2 = M.mqa_logits(W.Fp4Logits(**{**w.__dict__, "kv_fused": kv}))
    assert np.all(np.isnan(o2[: w.n, 3]))
    mask = np.ones_like(out, dtype=bool)
    mask[: w.n, 3] = False
    assert np.array_equal(o2[mask], out[mask])
